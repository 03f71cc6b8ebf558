"""The allocation-free forward entry point of the fused LM-head variant.

Some callers cannot allocate device memory when they need the loss: a serving or scoring
process that has given all of its device memory to its own pool (a KV cache, a caching
allocator) cannot cudaMalloc a workspace without failing or shrinking that pool, and some code
paths must not risk the device synchronisation cudaMalloc / cudaFree can cause. For them the
library keeps the forward pass's scratch in a fixed device array of its own.

This test calls that entry point through the C ABI twice in a row, with different shapes and
inputs (so the second call runs over whatever the first left in the shared array), and checks
each result against the workspace entry point's forward pass and against the float64 oracle,
within the per-token tolerances the other parity tests use. The file is named to be collected
last.
"""
import numpy as np
import pytest
import torch

from oracle import loss as OL
from rl_post_token_gb300 import _lib
from rl_post_token_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built(grpo_lib):
    assert torch.cuda.is_available()
    return grpo_lib


def _inputs(T, V, Hd, seed, with_old):
    wl = W.make_workload("lmhead", seed=seed, rows=4, tokens=T, V=V, H=Hd)
    h, Wt = W.make_lmhead_inputs(wl, DEV)
    rng = np.random.default_rng(seed)
    mask = wl.mask.copy()
    mask[rng.random(T) < 0.2] = 0
    adv = rng.choice([-1.5, -0.4, 0.6, 1.8], T).astype(np.float32)
    old = (rng.normal(-12.0, 1.0, T)).astype(np.float32) if with_old else None
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    return wl, h, Wt, t(wl.target), t(old), t(adv), t(mask), adv, mask, old


def _outputs(T):
    return (torch.full((T,), -7.0, device=DEV), torch.full((T,), -7.0, device=DEV), _lib.new_step_acc(DEV))


def test_noalloc_forward_matches_workspace_entry_point():
    cases = [(512, 8192, 128, 1, False), (300, 151936, 256, 2, True)]
    for T, V, Hd, seed, with_old in cases:
        wl, h, Wt, tgt, old, adv_d, mask_d, adv, mask, old_h = _inputs(T, V, Hd, seed, with_old)
        N = max(int(mask.sum()), 1)

        loss_r, logp_r, acc_r = _outputs(T)
        ws = torch.empty(_lib.grpo_lmhead_workspace_size(T, V, Hd), dtype=torch.uint8, device=DEV)
        _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, tgt, old, adv_d, mask_d, wl.eps, 1.0 / N, None, None,
                                      loss_r, logp_r, acc_r, ws)
        loss_n, logp_n, acc_n = _outputs(T)
        _lib.grpo_lmhead_forward_noalloc(h, Wt, tgt, old, adv_d, mask_d, wl.eps, 1.0 / N, loss_n, logp_n, acc_n)
        torch.cuda.synchronize()

        lr, pr = loss_r.double().cpu().numpy(), logp_r.double().cpu().numpy()
        ln, pn = loss_n.double().cpu().numpy(), logp_n.double().cpu().numpy()
        assert np.all(np.abs(pn - pr) <= 1e-5 * np.maximum(1.0, np.abs(pr)))
        assert np.all(np.abs(ln - lr) <= 1e-5 * np.abs(lr) + 1e-7 * np.abs(adv))
        res_r = _lib.grpo_finish_step(acc_r, loss_r, expected_N=int(mask.sum()))
        res_n = _lib.grpo_finish_step(acc_n, loss_n, expected_N=int(mask.sum()))
        for k in ("n_valid", "n_clipped", "n_nonfinite", "n_tokens", "status", "kernel_flags"):
            assert res_n[k] == res_r[k], k
        assert res_n["status"] == 0
        assert abs(res_n["loss"] - res_r["loss"]) <= 1e-5 * max(abs(res_r["loss"]), float(np.mean(np.abs(lr))))
        # and against the float64 oracle, token by token
        hb = h.view(torch.int16).cpu().numpy().view(np.uint16)
        wb = Wt.view(torch.int16).cpu().numpy().view(np.uint16)
        ref = OL.lmhead_fwd_bwd(hb, wb, wl.target, old_h, adv, mask, wl.eps, scale=1.0 / N, want_dw=False)
        m = mask.astype(bool)
        assert np.all(np.abs(pn[m] - ref["logp_tok"][m]) <= 1e-5 * np.maximum(1.0, np.abs(ref["logp_tok"][m])))
        assert np.all(np.abs(ln - ref["loss_tok"]) <= 1e-5 * np.abs(ref["loss_tok"]) + 1e-7 * np.abs(adv))
        assert np.all(pn[~m] == 0) and np.all(ln[~m] == 0)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    cap = _lib.grpo_lmhead_forward_noalloc_max_scratch()
    assert cap == 16 << 20
    T, V, Hd = 8192, 151936, 128  # needs ~39 MB of scratch
    h = torch.zeros((T, Hd), dtype=torch.bfloat16, device=DEV)
    Wt = torch.zeros((V, Hd), dtype=torch.bfloat16, device=DEV)
    i = torch.zeros(T, dtype=torch.int32, device=DEV)
    f = torch.zeros(T, device=DEV)
    m = torch.ones(T, dtype=torch.uint8, device=DEV)
    with pytest.raises(_lib.GrpoError) as e:
        _lib.grpo_lmhead_forward_noalloc(h, Wt, i, None, f, m, 0.2, 1.0, f, f, _lib.new_step_acc(DEV))
    assert e.value.code == _lib.ERR_CAPACITY
