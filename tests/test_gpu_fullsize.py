"""Full-size batches in the launch configuration the benchmark times (the same planner, chunk
loop and kernels), checked against the oracle on sampled token rows and by properties over
every row:
* sampled rows: per-token loss and log-prob, and the whole dlogits row, against the float64
  oracle with the per-token and dlogits bars of the smaller parity tests;
* every row: finite dlogits; each valid row's dlogits sum to ~0 (softmax and one-hot both sum
  to one); masked and padding rows exactly zero; per-step N equals the planner's N;
* the forward-only pass over the same batch: every token's loss and log-prob the bits of the
  full pass;
* the headline batch streamed from pinned host memory (the host entry point): the device run's
  bits.

pi_old here is target logit - 12 + N(0, 0.05): a plain input recipe (no log-softmax) that puts
the ratio far below 1, so tokens with A < 0 take the clipped branch and tokens with A > 0 the
unclipped one, both at full size."""
import numpy as np
import pytest
import torch

from oracle import loss as OL
from rl_post_token_gb300 import _lib
from rl_post_token_gb300 import step as S
from rl_post_token_gb300 import workloads as W

from tests import _gpu_helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built(grpo_lib):
    assert torch.cuda.is_available()
    return grpo_lib


def _host_row(t):
    return W.logits_to_host(t.unsqueeze(0))[0]


@pytest.mark.parametrize("name", ["qwen_step", "dynamic", "compaction"])
def test_full_size_batch(name):
    wl = W.make_workload(name, seed=0)
    bp = S.plan_batch(wl.plan, wl.row_len, wl.row_valid, wl.seg_counts)
    Te, T = bp.exec_tokens, wl.T
    logits = W.make_logits(wl, DEV, rows=Te)
    tok_src = None if bp.tok_src is None else bp.tok_src
    src = np.arange(Te) if tok_src is None else tok_src
    # pi_old from the target logit of each exec row's input token (valid rows only matter)
    tgt_exec = np.where(src >= 0, wl.target[np.where(src >= 0, src, -1 - src)], 0)
    zy = logits[torch.arange(Te, device=DEV), torch.from_numpy(tgt_exec.astype(np.int64)).to(DEV)].float().cpu().numpy()
    old = np.zeros(T, np.float32)
    ok = src >= 0
    old[src[ok]] = zy[ok] - 12.0 + wl.old_noise[src[ok]]
    adv = np.random.default_rng(1).choice([-1.5, -0.3, 0.4, 1.2], T).astype(np.float32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    dl = torch.empty_like(logits)
    loss = torch.full((T,), -7.0, device=DEV)
    logp = torch.full((T,), -7.0, device=DEV)
    accs = torch.zeros(bp.n_steps * _lib.ACC_BYTES, dtype=torch.uint8, device=DEV)
    S.run_batch(bp, logits=logits, dlogits=dl, target=t(wl.target), old_logp=t(old), mask=t(wl.mask),
                adv_tok=t(adv), loss_tok=loss, logp_tok=logp, accs=accs, clip_eps=wl.eps,
                tok_src=None if tok_src is None else t(tok_src), V=wl.V)
    torch.cuda.synchronize()
    res = S.read_results(accs, bp.n_steps)
    for s, r in enumerate(res):
        assert r["status"] == 0 and r["n_valid"] == bp.plan["step_valid_tokens"][s]

    # the same batch forward only (the pi_old ahead pass, on its own streaming kernel): every
    # token's loss and log-prob, and every step's result, are the bits of the full pass
    loss_f = torch.full((T,), -7.0, device=DEV)
    logp_f = torch.full((T,), -7.0, device=DEV)
    accs_f = torch.zeros_like(accs)
    S.run_batch(bp, logits=logits, dlogits=None, target=t(wl.target), old_logp=t(old), mask=t(wl.mask),
                adv_tok=t(adv), loss_tok=loss_f, logp_tok=logp_f, accs=accs_f, clip_eps=wl.eps,
                tok_src=None if tok_src is None else t(tok_src), V=wl.V)
    torch.cuda.synchronize()
    assert torch.equal(loss_f.view(torch.int32), loss.view(torch.int32))
    assert torch.equal(logp_f.view(torch.int32), logp.view(torch.int32))
    res_f = S.read_results(accs_f, bp.n_steps)
    for a, b in zip(res_f, res):
        for k in ("loss", "n_valid", "n_clipped", "n_nonfinite", "n_tokens", "status"):
            assert a[k] == b[k], k

    if name == "qwen_step":
        # the same batch streamed from pinned host memory through the host entry point (the
        # bench's e2e path): the device run's bits, at full size
        lh = logits.cpu().pin_memory()
        staging = torch.empty(2 * 1024 * logits.stride(0) * logits.element_size(), dtype=torch.uint8, device=DEV)
        dl_h = torch.empty_like(logits)
        loss_h = torch.full((T,), -7.0, device=DEV)
        logp_h = torch.full((T,), -7.0, device=DEV)
        accs_h = torch.zeros_like(accs)
        S.run_batch(bp, logits=None, logits_host=lh, staging=staging, block_rows=1024, copy_stream=torch.cuda.Stream(),
                    dlogits=dl_h, target=t(wl.target), old_logp=t(old), mask=t(wl.mask), adv_tok=t(adv),
                    loss_tok=loss_h, logp_tok=logp_h, accs=accs_h, clip_eps=wl.eps,
                    tok_src=None if tok_src is None else t(tok_src), V=wl.V)
        torch.cuda.synchronize()
        assert torch.equal(dl_h.view(torch.int16), dl.view(torch.int16))
        assert torch.equal(loss_h.view(torch.int32), loss.view(torch.int32))
        assert torch.equal(logp_h.view(torch.int32), logp.view(torch.int32))
        assert S.read_results(accs_h, bp.n_steps) == res
        del lh, dl_h

    # sampled exec rows: the first and last of every chunk plus a seeded handful
    rng = np.random.default_rng(2)
    pick = set()
    for c in range(bp.plan["n_chunks"]):
        a, b = int(bp.exec_tok_off[c]), int(bp.exec_tok_off[c + 1])
        if b > a:
            pick.update([a, b - 1])
    pick.update(rng.integers(0, Te, 12).tolist())
    pick = sorted(pick)[:48]
    step_of = np.zeros(Te, np.int64)
    for s, (e0, e1) in enumerate(bp.step_exec_range):
        step_of[e0:e1] = s
    lg, lp = H.to_f64(loss), H.to_f64(logp)
    for e in pick:
        i = int(src[e])
        scale = 1.0 / max(int(bp.plan["step_valid_tokens"][step_of[e]]), 1)
        got = dl[e].float().cpu().numpy().astype(np.float64)
        if i < 0:  # padding row
            assert np.all(got == 0)
            continue
        z = OL.as_f64(_host_row(logits[e]))
        lt, lpv, r, cl, dz = OL.token_objective(z, int(wl.target[i]), float(old[i]), float(adv[i]),
                                                int(wl.mask[i]), wl.eps, scale)
        ref = {"loss_tok": np.array([lt]), "logp_tok": np.array([lpv])}
        H.assert_tokens_close(lg[[i]], lp[[i]], ref, adv[[i]], wl.mask[[i]])
        coef = 0.0 if (cl or not wl.mask[i]) else float(adv[i]) * r * scale
        H.assert_dlogits_close(got[None, :], dz[None, :], "bf16", target=np.array([wl.target[i]]),
                               coef=np.array([coef]))

    # properties over every row, in blocks
    valid_exec = torch.from_numpy((src >= 0) & (wl.mask[np.where(src >= 0, src, 0)] != 0)).to(DEV)
    for a in range(0, Te, 4096):
        blk = dl[a:a + 4096].float()
        assert torch.isfinite(blk).all()
        rs = blk.sum(1).abs()
        mag = blk.abs().sum(1)
        v = valid_exec[a:a + 4096]
        assert torch.all(rs[v] <= 2e-2 * mag[v] + 1e-12)
        assert torch.all(mag[~v] == 0)


@pytest.mark.parametrize("dtype, V", [("bf16", 151936), ("f32", 151936)])
def test_forward_only_repeated_calls_give_the_training_pass_bits(dtype, V):
    # The forward-only kernel's cross-CTA exchange (partials sent by asynchronous DSMEM stores,
    # combined by one warp of the cluster's first CTA) against the training pass, 40 calls in a
    # row at the product vocabulary: every call's loss and log-prob must be the training pass's
    # bits, so a partial read before it landed, or a buffer reused while still being read,
    # would show as a mismatch.
    T = 1024 if dtype == "bf16" else 512
    wl = W.make_workload("tiny", rows=8, positions=T // 8, valid_lo=0, V=V, dtype=dtype, seed=77, std=3.0)
    case = H.Case(wl, old_mode="none")
    lg = case.logits
    adv = torch.from_numpy(np.random.default_rng(5).normal(0, 1, wl.T).astype(np.float32)).to(DEV)
    old = torch.from_numpy(np.random.default_rng(6).normal(-12, 1, wl.T).astype(np.float32)).to(DEV)
    dl = torch.empty_like(lg)
    loss_t, logp_t = torch.empty(wl.T, device=DEV), torch.empty(wl.T, device=DEV)
    _lib.grpo_logprob_loss_fwd_bwd(lg, case.d_target, old, adv, case.d_mask, wl.eps, 1.0, dl, loss_t, logp_t,
                                   _lib.new_step_acc(DEV))
    torch.cuda.synchronize()
    loss_f, logp_f = torch.empty(wl.T, device=DEV), torch.empty(wl.T, device=DEV)
    for k in range(40):
        loss_f.fill_(7.0)
        logp_f.fill_(7.0)
        acc = _lib.new_step_acc(DEV)
        _lib.grpo_logprob_loss_fwd_bwd(lg, case.d_target, old, adv, case.d_mask, wl.eps, 1.0, None, loss_f, logp_f,
                                       acc)
        torch.cuda.synchronize()
        assert torch.equal(loss_f.view(torch.int32), loss_t.view(torch.int32)), k
        assert torch.equal(logp_f.view(torch.int32), logp_t.view(torch.int32)), k
        res = _lib.grpo_finish_step(acc, loss_f)
        assert res["kernel_flags"] == 0 and res["n_valid"] == int(wl.mask.sum()), k
