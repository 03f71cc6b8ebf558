"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random inputs; it holds none of the method's arithmetic (no
log-softmax, no ratio, no advantage). The library and the float64 oracle are both fed from
here. pi_old is not drawn directly: a workload carries ``old_noise``, and the caller forms
``old_logp = reference_logp + old_noise`` from a reference log-prob of its own (the oracle in
the tests, the library's forward-only ahead pass in the benchmark).

Draw order from ``numpy.random.default_rng(seed)``: row lengths -> valid lengths -> rewards ->
targets -> old-logp noise. Logits come from a second stream: numpy ``default_rng(seed + 1)``
(float32 normal, rounded to bfloat16 to nearest even) when small, else a seeded
``torch.Generator`` on the target device (normal, rounded by torch). Tests always read the
logits actually handed to the GPU back to the host before giving them to the oracle.

Workloads (the pages measure on no public benchmark; these stand in for the Qwen3-VL-2B runs
of "Sizing mini-batches and micro-batches", *The problem*, and for the worked examples):

* ``tiny``       8 prompts x 4 rollouts, 64 positions per row (padded layout), mask prefix
                 lengths uniform in [16, 64], V = 512 float32 logits ~ N(0, 2), rewards
                 Bernoulli(0.5), mini 16, micro 8 (the 2x2 loop).
* ``qwen_step``  8 x 4 rollouts, completion lengths uniform in [128, 2048] (packed), every
                 completion token valid, V = 151936 bf16 logits ~ N(0, 3), rewards
                 Bernoulli(0.3), mini 16, micro 8.
* ``dynamic``    16 x 8 rollouts, lengths clamp(round(exp(N(ln 700, 0.6^2))), 1, 2048),
                 V = 151936 bf16 ~ N(0, 3), rewards Bernoulli(0.3), one optimizer step,
                 token-budget bins of 16384 tokens by attention workload, small bins at the
                 ends.
* ``compaction`` 3 prompts x 2 generations with segments {1,3}, {2,5}, {1,1}, 1024 tokens
                 per row, V = 151936 bf16 ~ N(0, 3), rewards Bernoulli(0.5), Q = 4 x lcm(1, 1).
* ``lmhead``     16384 tokens (8 x 2048), hidden [16384, 2048] bf16 ~ N(0, 1), W [151936, 2048]
                 bf16 ~ N(0, 0.02); other fields as ``qwen_step``.
pi_old noise is N(0, 0.05) everywhere unless ``old_sigma`` is overridden (0.5 is the stress
case in which the clip binds often).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

V_QWEN = 151936
HOST_LOGITS_MAX_ELEMS = 64 * 1024 * 1024  # above this, logits are drawn on the device


@dataclass
class Workload:
    name: str
    seed: int
    V: int
    dtype: str                 # "f32" or "bf16"
    logit_std: float
    eps: float
    group_size: int
    plan: dict                 # planner fields (same names as the C struct)
    row_len: np.ndarray        # int32 [rows]: logits rows per input row
    row_valid: np.ndarray      # int32 [rows]: mask=1 positions per input row
    mask: np.ndarray           # uint8 [T]: response mask in input token order
    target: np.ndarray         # int32 [T]: sampled token ids
    rewards: np.ndarray        # float32 [rollouts]
    old_noise: np.ndarray      # float32 [T]: pi_old = reference logp + old_noise
    seg_counts: Optional[np.ndarray] = None  # int32 [rollouts] (compaction)
    row_rollout: Optional[np.ndarray] = None  # int32 [rows]: rollout of each input row
    extra: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.row_len.sum())

    @property
    def n_rollouts(self) -> int:
        return int(self.rewards.shape[0])

    @property
    def tok_off(self) -> np.ndarray:
        off = np.zeros(self.row_len.shape[0] + 1, np.int64)
        np.cumsum(self.row_len, out=off[1:])
        return off

    @property
    def n_valid(self) -> int:
        return int(self.mask.astype(np.int64).sum())

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


def _finish(name, seed, rng, V, dtype, std, G, plan, row_len, row_valid, rewards_p, n_rollouts,
            old_sigma, eps=0.2, seg_counts=None, row_rollout=None, padded_mask=False):
    row_len = np.asarray(row_len, np.int32)
    row_valid = np.asarray(row_valid, np.int32)
    rewards = (rng.random(n_rollouts) < rewards_p).astype(np.float32)
    T = int(row_len.sum())
    target = rng.integers(0, V, T, dtype=np.int64).astype(np.int32)
    old_noise = rng.normal(0.0, old_sigma, T).astype(np.float32)
    mask = np.zeros(T, np.uint8)
    off = 0
    for L, v in zip(row_len, row_valid):
        mask[off:off + v] = 1   # completion positions first, padding after (prefix mask)
        off += L
    if row_rollout is None:
        row_rollout = np.arange(row_len.shape[0], dtype=np.int32)
    return Workload(name=name, seed=seed, V=V, dtype=dtype, logit_std=std, eps=eps, group_size=G,
                    plan=plan, row_len=row_len, row_valid=row_valid, mask=mask, target=target,
                    rewards=rewards, old_noise=old_noise,
                    seg_counts=None if seg_counts is None else np.asarray(seg_counts, np.int32),
                    row_rollout=np.asarray(row_rollout, np.int32))


def make_workload(name: str, seed: int = 0, old_sigma: float = 0.05, **ov) -> Workload:
    """Build one workload. Overrides (``V``, ``rows``, ``len_lo``, ``len_hi``, ``dtype``,
    ``mini``, ``micro``, ``max_token_len``, ...) shrink it for parity tests."""
    rng = np.random.default_rng(seed)
    if name == "tiny":
        B = ov.get("rows", 32)
        P = ov.get("positions", 64)
        V = ov.get("V", 512)
        row_len = np.full(B, P, np.int32)
        row_valid = rng.integers(ov.get("valid_lo", 16), P + 1, B)
        plan = dict(batch=B, mini=ov.get("mini", 16), micro=ov.get("micro", 8), group_size=4)
        return _finish(name, seed, rng, V, ov.get("dtype", "f32"), ov.get("std", 2.0), 4, plan,
                       row_len, row_valid, 0.5, B, old_sigma)
    if name == "qwen_step":
        B = ov.get("rows", 32)
        V = ov.get("V", V_QWEN)
        row_len = rng.integers(ov.get("len_lo", 128), ov.get("len_hi", 2048) + 1, B)
        plan = dict(batch=B, mini=ov.get("mini", 16), micro=ov.get("micro", 8), group_size=4)
        return _finish(name, seed, rng, V, ov.get("dtype", "bf16"), ov.get("std", 3.0), 4, plan,
                       row_len, row_len, 0.3, B, old_sigma)
    if name == "dynamic":
        B = ov.get("rows", 128)
        V = ov.get("V", V_QWEN)
        cap = ov.get("len_hi", 2048)
        row_len = np.clip(np.round(np.exp(rng.normal(np.log(ov.get("median", 700)), 0.6, B))), 1, cap)
        row_len = row_len.astype(np.int32)
        plan = dict(batch=B, mini=ov.get("mini", 0), micro=0, group_size=8, dynamic=1,
                    max_token_len=ov.get("max_token_len", 16384), workload=1, balance_ends=1)
        return _finish(name, seed, rng, V, ov.get("dtype", "bf16"), ov.get("std", 3.0), 8, plan,
                       row_len, row_len, 0.3, B, old_sigma)
    if name == "compaction":
        V = ov.get("V", V_QWEN)
        segs = ov.get("segments", [[1, 3], [2, 5], [1, 1]])
        G = len(segs[0])
        seg = [s for grp in segs for s in grp]
        n_rows = sum(seg)
        Lrow = ov.get("row_tokens", 1024)
        row_len = np.full(n_rows, Lrow, np.int32)
        row_rollout = np.repeat(np.arange(len(seg), dtype=np.int32), seg)
        plan = dict(batch=len(seg), mini=0, micro=1, group_size=G, compaction=1, n_gpus=4,
                    logprob_batch=1)
        return _finish(name, seed, rng, V, ov.get("dtype", "bf16"), ov.get("std", 3.0), G, plan,
                       row_len, row_len, 0.5, len(seg), old_sigma, seg_counts=seg,
                       row_rollout=row_rollout)
    if name == "lmhead":
        B = ov.get("rows", 8)
        Lrow = ov.get("row_tokens", 2048)
        V = ov.get("V", V_QWEN)
        row_len = np.full(B, Lrow, np.int32)
        if "tokens" in ov:  # T tokens over B rows, the last row taking the remainder
            row_len[:] = ov["tokens"] // B
            row_len[-1] = ov["tokens"] - (B - 1) * (ov["tokens"] // B)
        plan = dict(batch=B, mini=0, micro=0, group_size=4)
        wl = _finish(name, seed, rng, V, "bf16", 0.0, 4, plan, row_len, row_len, 0.3, B, old_sigma)
        wl.extra.update(H=ov.get("H", 2048), h_std=1.0, w_std=0.02)
        return wl
    raise ValueError(f"unknown workload {name}")


def bf16_round_bits(x32: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (input encoding only)."""
    u = x32.astype(np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def make_logits(wl: Workload, device="cpu", rows: Optional[int] = None, torch_dtype=None):
    """Logits [T, V] for a workload as a torch tensor on ``device``.

    Small workloads draw on the host with numpy (so the values do not depend on the device);
    large ones draw with a seeded ``torch.Generator`` on ``device`` in row blocks."""
    import torch

    T = wl.T if rows is None else rows
    V = wl.V
    tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    if T * V <= HOST_LOGITS_MAX_ELEMS:
        rng = np.random.default_rng(wl.seed + 1)
        x = (rng.standard_normal((T, V), dtype=np.float32) * np.float32(wl.logit_std))
        if wl.dtype == "f32":
            return torch.from_numpy(x).to(device)
        bits = bf16_round_bits(x)
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device)
    out = torch.empty((T, V), dtype=tdt, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed + 1)
    blk = max(1, (256 * 1024 * 1024) // (4 * V))
    for a in range(0, T, blk):
        b = min(T, a + blk)
        tmp = torch.randn((b - a, V), generator=g, device=device, dtype=torch.float32)
        tmp.mul_(wl.logit_std)
        out[a:b].copy_(tmp)
    return out


def logits_to_host(t) -> np.ndarray:
    """Read logits back for the oracle: float32 values or bfloat16 bit patterns (uint16)."""
    import torch

    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def make_lmhead_inputs(wl: Workload, device="cpu"):
    """Hidden states h [T, H] ~ N(0, 1) and output embedding W [V, H] ~ N(0, 0.02), bf16, as
    torch tensors on ``device`` (numpy when small, a seeded device generator when large)."""
    import torch

    T, V, H = wl.T, wl.V, wl.extra["H"]
    out = []
    for k, (rows, std) in enumerate([(T, wl.extra["h_std"]), (V, wl.extra["w_std"])]):
        if rows * H <= HOST_LOGITS_MAX_ELEMS:
            rng = np.random.default_rng(wl.seed + 11 + k)
            bits = bf16_round_bits(rng.standard_normal((rows, H), dtype=np.float32) * np.float32(std))
            out.append(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(device))
        else:
            g = torch.Generator(device=device)
            g.manual_seed(wl.seed + 11 + k)
            t = torch.empty((rows, H), dtype=torch.bfloat16, device=device)
            blk = max(1, (256 * 1024 * 1024) // (4 * H))
            for a in range(0, rows, blk):
                b = min(rows, a + blk)
                t[a:b].copy_(torch.randn((b - a, H), generator=g, device=device) * std)
            out.append(t)
    return out[0], out[1]
