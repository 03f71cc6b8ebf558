"""The C ABI from plain C programs, with no Python or torch in their process.
tests/c_abi/loss_step.c (the row pass) and tests/c_abi/lmhead_step.c (the fused LM-head step)
are compiled with gcc against include/grpo.h, libgrpo.so and the CUDA runtime, and run on
seeded inputs. Their outputs (per-token loss and log-prob, dlogits or d_h and dW, the step
result) must equal the Python binding's on the same inputs, bit for bit."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from rl_post_token_gb300 import _lib
from rl_post_token_gb300 import workloads as W

from tests import _gpu_helpers as H

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    pytest.skip("CUDA toolkit headers not found")


def _compile(out_dir, name="loss_step"):
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("gcc not found")
    cuda = _cuda_home()
    pkg = os.path.join(ROOT, "rl_post_token_gb300")
    exe = os.path.join(out_dir, name)
    cmd = [gcc, "-std=c11", "-O2", "-Wall", f"-I{ROOT}/include", f"-I{cuda}/include",
           os.path.join(ROOT, "tests", "c_abi", name + ".c"), "-o", exe, f"-L{pkg}", "-lgrpo",
           f"-L{cuda}/lib64", "-lcudart", f"-Wl,-rpath,{pkg}", f"-Wl,-rpath,{cuda}/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_plain_c_client_matches_the_binding(grpo_lib, tmp_path):
    assert torch.cuda.is_available()
    exe = _compile(str(tmp_path))
    wl = W.make_workload("tiny", rows=8, positions=16, valid_lo=0, V=32776, dtype="bf16", seed=99, std=2.0)
    case = H.Case(wl)
    T, V = case.logits.shape
    scale = np.float32(1.0 / max(int(wl.mask.sum()), 1))
    inp, outp = os.path.join(str(tmp_path), "in.bin"), os.path.join(str(tmp_path), "out.bin")
    with open(inp, "wb") as f:
        f.write(np.int64(T).tobytes() + np.int64(V).tobytes())
        f.write(np.float32(wl.eps).tobytes() + scale.tobytes())
        f.write(case.logits.view(torch.int16).cpu().numpy().astype(np.uint16).tobytes())
        f.write(np.asarray(wl.target, np.int32).tobytes() + np.asarray(case.old, np.float32).tobytes())
        f.write(np.asarray(case.adv_tok, np.float32).tobytes() + np.asarray(wl.mask, np.uint8).tobytes())
    r = subprocess.run([exe, inp, outp], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = open(outp, "rb").read()
    o = 0
    status = int(np.frombuffer(raw, np.int32, 1, o)[0]); o += 4
    c_loss = np.frombuffer(raw, np.float32, T, o); o += 4 * T
    c_logp = np.frombuffer(raw, np.float32, T, o); o += 4 * T
    c_dz = np.frombuffer(raw, np.uint16, T * V, o); o += 2 * T * V
    c_res_loss = float(np.frombuffer(raw, np.float64, 1, o)[0]); o += 8
    c_n_valid, c_n_clipped = (int(x) for x in np.frombuffer(raw, np.int64, 2, o))

    # the binding, same inputs
    dl = torch.empty_like(case.logits)
    loss, logp = torch.empty(T, device=DEV), torch.empty(T, device=DEV)
    acc = _lib.new_step_acc(DEV)
    _lib.grpo_logprob_loss_fwd_bwd(case.logits, case.d_target, case.d_old, case.d_adv, case.d_mask, wl.eps,
                                   float(scale), dl, loss, logp, acc)
    res = _lib.grpo_finish_step(acc, loss)
    assert status == res["status"] == 0
    assert np.array_equal(c_loss.view(np.uint32), loss.cpu().numpy().view(np.uint32))
    assert np.array_equal(c_logp.view(np.uint32), logp.cpu().numpy().view(np.uint32))
    assert np.array_equal(c_dz, dl.view(torch.int16).cpu().numpy().astype(np.uint16).ravel())
    assert c_res_loss == res["loss"] and c_n_valid == res["n_valid"] and c_n_clipped == res["n_clipped"]


def test_plain_c_lmhead_client_matches_the_binding(grpo_lib, tmp_path):
    assert torch.cuda.is_available()
    exe = _compile(str(tmp_path), "lmhead_step")
    T, V, Hd = 300, 3000, 192
    wl = W.make_workload("lmhead", seed=61, rows=4, tokens=T, V=V, H=Hd)
    h, Wt = W.make_lmhead_inputs(wl, DEV)
    rng = np.random.default_rng(61)
    mask = wl.mask.copy()
    mask[rng.random(T) < 0.2] = 0
    adv = rng.normal(0, 1, T).astype(np.float32)
    old = rng.normal(-9, 1, T).astype(np.float32)
    ref = (old + rng.normal(0, 0.3, T)).astype(np.float32)
    scale = np.float32(1.0 / max(int(mask.sum()), 1))
    inp, outp = os.path.join(str(tmp_path), "in.bin"), os.path.join(str(tmp_path), "out.bin")
    with open(inp, "wb") as f:
        f.write(np.int64(T).tobytes() + np.int64(V).tobytes() + np.int64(Hd).tobytes())
        f.write(np.float32(wl.eps).tobytes() + scale.tobytes())
        f.write(h.view(torch.int16).cpu().numpy().astype(np.uint16).tobytes())
        f.write(Wt.view(torch.int16).cpu().numpy().astype(np.uint16).tobytes())
        f.write(np.asarray(wl.target, np.int32).tobytes() + old.tobytes() + adv.tobytes() + mask.tobytes())
        f.write(ref.tobytes())
    r = subprocess.run([exe, inp, outp], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = open(outp, "rb").read()
    o = 0
    steps = []
    for _ in range(2):  # the plain step, then the one with the regularisers and the flag
        status = int(np.frombuffer(raw, np.int32, 1, o)[0]); o += 4
        c_loss = np.frombuffer(raw, np.float32, T, o); o += 4 * T
        c_logp = np.frombuffer(raw, np.float32, T, o); o += 4 * T
        c_dh = np.frombuffer(raw, np.float32, T * Hd, o); o += 4 * T * Hd
        c_dw = np.frombuffer(raw, np.float32, V * Hd, o); o += 4 * V * Hd
        c_res_loss = float(np.frombuffer(raw, np.float64, 1, o)[0]); o += 8
        c_n_valid, c_n_clipped = (int(x) for x in np.frombuffer(raw, np.int64, 2, o)); o += 16
        steps.append((status, c_loss, c_logp, c_dh, c_dw, c_res_loss, c_n_valid, c_n_clipped))
    c_ent = np.frombuffer(raw, np.float32, T, o)

    # the binding, same inputs
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    ent = torch.empty(T, device=DEV)
    for k, (status, c_loss, c_logp, c_dh, c_dw, c_res_loss, c_n_valid, c_n_clipped) in enumerate(steps):
        d_h = torch.empty((T, Hd), device=DEV)
        dW = torch.empty((V, Hd), device=DEV)
        loss, logp = torch.empty(T, device=DEV), torch.empty(T, device=DEV)
        acc = _lib.new_step_acc(DEV)
        ws = torch.empty(_lib.grpo_lmhead_workspace_size(T, V, Hd), dtype=torch.uint8, device=DEV)
        terms = None if k == 0 else dict(kl_kind=_lib.KL_K3, kl_coef=0.1, ref_logp=t(ref), ent_coef=0.02,
                                         entropy_tok=ent)
        _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, t(wl.target), t(old), t(adv), t(mask), wl.eps, float(scale), d_h, dW,
                                      loss, logp, acc, ws, terms=terms, skip_masked=k == 1)
        res = _lib.grpo_finish_step(acc, loss)
        assert status == res["status"] == 0
        for got, want in ((c_loss, loss), (c_logp, logp), (c_dh, d_h), (c_dw, dW)):
            assert np.array_equal(got.view(np.uint32), want.cpu().numpy().ravel().view(np.uint32)), k
        assert c_res_loss == res["loss"] and c_n_valid == res["n_valid"] and c_n_clipped == res["n_clipped"]
    assert np.array_equal(c_ent.view(np.uint32), ent.cpu().numpy().view(np.uint32))
