"""Child process of tests/test_gpu_threads.py (run as ``python -m tests._threads_child`` from
the repository root, so that the library's per-kernel launch caches start empty).

Several host threads, each on its own CUDA stream with its own outputs, call the library at
the same time: every row-pass instance (plain, forward-only, with KL / entropy / weights, the
L2 kernel for short rows, both logit types), the row pass over pinned host logits, and both
LM-head backward paths, each call followed by its step finish. Each result (per-token outputs,
gradients, the finished step's result) must equal, bit for bit, the same call made alone
afterwards. Prints ``THREADS_OK <n>`` (n
compared buffers) and exits 0, or prints the first mismatch and exits 1."""
import sys
import threading

import numpy as np
import torch

from rl_post_token_gb300 import _lib
from rl_post_token_gb300 import workloads as W

DEV = "cuda"
N_THREADS = 4
REPS = 3


def _bits(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    if t.dtype == torch.float32:
        return t.view(torch.int32)
    return t


class RowCase:
    """One row-pass call: inputs shared by all threads, outputs made per caller."""

    def __init__(self, k, V, dtype, grad, terms):
        wl = W.make_workload("qwen_step", rows=4, len_lo=16, len_hi=28, V=V, dtype=dtype, seed=900 + k)
        self.logits = W.make_logits(wl, DEV)
        T = self.T = self.logits.shape[0]
        rng = np.random.default_rng(900 + k)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
        lse = np.log(V) + 4.5  # about the LSE of N(0, 3) logits
        self.target, self.mask = t(wl.target), t(wl.mask)
        a = rng.normal(0.0, 1.0, T).astype(np.float32)
        if k % 2:  # a third of the tokens without a gradient: the backward's live-token partition
            a[: T // 3] = 0.0
        self.adv = t(a)
        self.old = t((-lse + rng.normal(0.0, 1.0, T)).astype(np.float32))
        self.grad = grad
        self.terms = terms
        if terms is not None:
            self.ref = t((-lse + rng.normal(0.0, 1.0, T)).astype(np.float32))
            self.w_tok = t(rng.uniform(0.5, 2.0, T).astype(np.float32))

    def outputs(self):
        T = self.T
        # filled, so that an element no call writes compares equal too
        o = {"loss": torch.full((T,), -7.0, device=DEV), "logp": torch.full((T,), -7.0, device=DEV),
             "acc": _lib.new_step_acc(DEV)}
        if self.grad:
            o["dl"] = torch.full_like(self.logits, 7.0)
        if self.terms is not None and self.terms.get("ent_coef"):
            o["ent"] = torch.full((T,), -7.0, device=DEV)
        return o

    def call(self, o, stream):
        terms = None
        if self.terms is not None:
            terms = dict(self.terms)
            if terms.get("kl_kind"):
                terms["ref_logp"] = self.ref
            if terms.get("ent_coef"):
                terms["entropy_tok"] = o["ent"]
            if terms.get("w_tok"):
                terms["w_tok"] = self.w_tok
        _lib.grpo_logprob_loss_fwd_bwd(self.logits, self.target, self.old, self.adv, self.mask, 0.2,
                                       1.0 / 700, o.get("dl"), o["loss"], o["logp"], o["acc"],
                                       stream=stream, terms=terms)
        _lib.grpo_finish_step(o["acc"], o["loss"], sync=False, stream=stream)


class HostCase(RowCase):
    """The row pass over pinned host logits: each caller has its own staging buffer and copy
    stream (32-row blocks, so a call runs several blocks through the two halves)."""

    BLOCK = 32

    def __init__(self, k):
        super().__init__(k, W.V_QWEN, "bf16", True, None)
        self.host = self.logits.cpu().pin_memory()

    def outputs(self):
        o = super().outputs()
        o["_staging"] = torch.empty(2 * self.BLOCK * self.host.stride(0) * 2, dtype=torch.uint8, device=DEV)
        o["_copy"] = torch.cuda.Stream(DEV)
        return o

    def call(self, o, stream):
        _lib.grpo_logprob_loss_fwd_bwd_host(self.host, self.target, self.old, self.adv, self.mask, 0.2, 1.0 / 700,
                                            o["dl"], o["loss"], o["logp"], o["acc"], o["_staging"], self.BLOCK,
                                            stream=stream, copy_stream=o["_copy"])
        _lib.grpo_finish_step(o["acc"], o["loss"], sync=False, stream=stream)


class LmCase:
    def __init__(self, k):
        T, V, H = 384, 40000, 512
        wl = W.make_workload("lmhead", seed=950 + k, rows=4, tokens=T, V=V, H=H)
        self.h, self.W = W.make_lmhead_inputs(wl, DEV)
        rng = np.random.default_rng(950 + k)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
        self.target, self.mask = t(wl.target), t(wl.mask)
        a = rng.normal(0.0, 1.0, T).astype(np.float32)
        if k % 2:  # a third of the tokens without a gradient: the backward's live-token partition
            a[: T // 3] = 0.0
        self.adv = t(a)
        self.T, self.V, self.H = T, V, H
        self.ws_bytes = _lib.grpo_lmhead_workspace_size(T, V, H)

    def outputs(self):
        T, V, H = self.T, self.V, self.H
        return {"d_h": torch.full((T, H), 7.0, device=DEV), "dW": torch.full((V, H), 7.0, device=DEV),
                "loss": torch.full((T,), -7.0, device=DEV), "logp": torch.full((T,), -7.0, device=DEV),
                "acc": _lib.new_step_acc(DEV), "_ws": torch.empty(self.ws_bytes, dtype=torch.uint8, device=DEV)}

    def call(self, o, stream):
        _lib.grpo_lmhead_loss_fwd_bwd(self.h, self.W, self.target, None, self.adv, self.mask, 0.2, 1.0 / 300,
                                      o["d_h"], o["dW"], o["loss"], o["logp"], o["acc"], o["_ws"],
                                      stream=stream)
        _lib.grpo_finish_step(o["acc"], o["loss"], sync=False, stream=stream)


def main():
    assert torch.cuda.is_available()
    _lib.lib()
    big = W.V_QWEN
    cases = [
        RowCase(0, big, "bf16", True, None),
        RowCase(1, big, "f32", True, None),
        RowCase(2, big, "bf16", False, None),  # forward only: the streaming kernel
        RowCase(3, big, "f32", False, None),
        RowCase(4, big, "bf16", True, dict(ent_coef=0.01)),
        RowCase(5, big, "bf16", True, dict(kl_kind=_lib.KL_K3, kl_coef=0.05, w_tok=True)),
        RowCase(6, big, "f32", True, dict(kl_kind=_lib.KL_K1, kl_coef=0.05, ent_coef=0.01, w_tok=True)),
        RowCase(7, 1000, "bf16", True, None),  # short rows: the L2 kernel
        RowCase(8, 4104, "f32", True, dict(ent_coef=0.01)),
        LmCase(9),
        LmCase(10),
        HostCase(11),  # logits in pinned host memory, streamed through a staging buffer
    ]
    streams = [torch.cuda.Stream(DEV) for _ in range(N_THREADS)]
    # per thread, case and repetition its own outputs (accumulators zeroed here, before any
    # call): nothing is shared between callers
    outs = [[[c.outputs() for _ in range(REPS)] for c in cases] for _ in range(N_THREADS)]
    torch.cuda.synchronize()
    barrier = threading.Barrier(N_THREADS)
    errors = []

    def worker(i):
        try:
            order = list(range(len(cases)))
            order = order[i:] + order[:i]  # every thread starts on a different instance
            barrier.wait()
            for r in range(REPS):
                for j in order:
                    cases[j].call(outs[i][j][r], streams[i])
            streams[i].synchronize()
        except Exception as e:  # reported by the main thread
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(N_THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    if errors:
        print("THREAD ERROR", errors[0])
        return 1

    alone = torch.cuda.Stream(DEV)
    n = 0
    for j, c in enumerate(cases):
        ref = c.outputs()
        torch.cuda.synchronize()  # the fresh accumulator's zeroing ran on another stream
        c.call(ref, alone)
        alone.synchronize()
        for i in range(N_THREADS):
            for r in range(REPS):
                got = outs[i][j][r]
                for key, want in ref.items():
                    if key.startswith("_"):
                        continue
                    a, b = _bits(got[key]), _bits(want)  # acc: the finish's result and divisor too
                    if not torch.equal(a, b):
                        print(f"MISMATCH case {j} thread {i} rep {r} output {key}")
                        return 1
                    n += 1
    print("THREADS_OK", n)
    return 0


if __name__ == "__main__":
    sys.exit(main())
