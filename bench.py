"""Benchmark: GRPO loss forward+backward, valid tokens/s at V = 151936 bf16, and the fraction of
the HBM roofline.

A "step" is one whole collected batch through the library: plan -> group advantage -> every
(mini, micro) chunk's loss forward+backward -> every optimizer step's finish. The default
workload is the Qwen3-VL-2B-shaped step (8 prompts x 4 rollouts, completion lengths uniform in
[128, 2048], V = 151936 bf16 logits ~ N(0, 3), mini 16, micro 8), synthetic and seeded; its
~10.6 GB of logits are larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload qwen_step|dynamic|compaction|tiny]

Under torchrun (N > 1) every rank runs its own batch (weak scaling, no collective on the
data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GRPO loss fwd+bwd valid tokens/s at V=151936 bf16; % of HBM roofline"
LMHEAD_METRIC = "GRPO loss fwd+bwd valid tokens/s, fused LM-head (V=151936, H=2048, bf16)"
UNIT = "valid tokens/s"
FALLBACK_HBM_GBS = 6800.0
# device code of the row-pass kernel (the profile records the combined hash of these files)
KERNEL_SRC = tuple(os.path.join(ROOT, "rl_post_token_gb300", "csrc", f)
                   for f in ("grpo_rowpass_kernels.cuh", "grpo_common.cuh"))


def _code_only(text: str) -> str:
    """The source without comments, trailing spaces or blank lines: what the compiler sees."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_sha256() -> str:
    """Hash of the row-pass kernels' device code (comments ignored), tying the committed ncu
    traffic figure to the code it was measured on."""
    h = hashlib.sha256()
    for f in KERNEL_SRC:
        h.update(_code_only(open(f, encoding="utf-8").read()).encode())
    return h.hexdigest()


WORKLOAD_TEXT = {
    "qwen_step": "Qwen3-VL-2B-shaped step: 8 prompts x 4 rollouts, completion lengths U[128,2048] "
                 "packed, V=151936 bf16 logits ~N(0,3), mini 16, micro 8, rewards Bernoulli(0.3), eps 0.2",
    "dynamic": "dynamic batching: 16 prompts x 8 rollouts, lognormal lengths (median 700, cap 2048), "
               "V=151936 bf16, token-budget bins of 16384 by attention workload, one optimizer step",
    "compaction": "context compaction: 3 prompts x 2 generations, segments {1,3},{2,5},{1,1}, 1024-token "
                  "rows, Q=4 -> 16 rows incl. 3 pad rows, V=151936 bf16, one step",
    "tiny": "tiny oracle check: 8 prompts x 4 rollouts, 64 positions, V=512 f32, mini 16, micro 8",
    "lmhead": "fused LM-head: hidden [16384, 2048] bf16 ~N(0,1) x W [151936, 2048] bf16 ~N(0,0.02), "
              "tcgen05 GEMM chunked over V feeding the online softmax, d_hidden and dW outputs (f32)",
}


# ---- distributed helpers (also exercised by the CPU gloo test) ---------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_timing(elapsed_s: float, units: float, world: int, device=None):
    """(max elapsed over ranks, sum of units over ranks)."""
    if world <= 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---- peaks, clocks, profiles --------------------------------------------------------------------

def bf16_peak(sustained: bool = True):
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained" if sustained else "bf16_tflops"]), "measured"
    except Exception:
        return (1700.0 if sustained else 1900.0), "fallback"


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str):
        self.path = path
        self.proc = None
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_index)], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def profiled_traffic():
    """Per-valid-token DRAM traffic of the row-pass kernel from the committed ncu figure
    (profiles/rowpass_qwen_step_traffic.json), or None when it is missing or was taken on a
    different kernel source."""
    path = os.path.join(ROOT, "profiles", "rowpass_qwen_step_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        tpv, sha = float(d["traffic_per_valid_token_bytes"]), str(d["kernel_source_sha256"])
    except (OSError, ValueError, KeyError):
        return None
    return tpv if kernel_source_sha256() == sha else None


# ---- oracle timing (CPU baseline and reference arm) ----------------------------------------------

def oracle_sample_rate(wl, n_tokens: int, budget_s: float, lt=None):
    """Time the float64 oracle on the first valid tokens of a host-generated sample of the
    workload, with the regularisers of ``lt`` (cli_terms' dict) when given. Returns (valid
    tokens/s, tokens timed, seconds)."""
    from oracle import loss as OL
    from rl_post_token_gb300 import workloads as W

    rows = min(wl.T, n_tokens)
    rng = np.random.default_rng(wl.seed + 7)
    x = rng.standard_normal((rows, wl.V), dtype=np.float32) * np.float32(wl.logit_std)
    logits = W.bf16_round_bits(x) if wl.dtype == "bf16" else x
    tgt, msk, adv = wl.target[:rows], wl.mask[:rows], np.where(np.arange(rows) % 2, 1.0, -1.0)
    ref = np.array([OL.log_softmax_row(OL.as_f64(logits[t]))[tgt[t]] for t in range(rows)])
    old = ref + wl.old_noise[:rows]
    kl_ref = ref + np.random.default_rng(wl.seed + 1).normal(0.0, 0.1, rows)
    wt = oracle_token_weights(wl, lt)
    done, t0 = 0, time.perf_counter()
    while True:
        for t in range(rows):
            tt = oracle_terms(lt, kl_ref[t])
            OL.token_objective(OL.as_f64(logits[t]), int(tgt[t]), float(old[t]), float(adv[t]),
                               int(msk[t]), wl.eps, float(wt[t]), True, tt)
            done += int(msk[t])
            if time.perf_counter() - t0 > budget_s:
                break
        if time.perf_counter() - t0 > budget_s or done == 0:
            break
    dt = time.perf_counter() - t0
    return done / dt, done, dt


def oracle_terms(lt, ref):
    """The oracle's ``terms`` dict for one token (None without regularisers)."""
    if lt is None or not (lt["kl_kind"] or lt["ent_coef"]):
        return None
    return {"kl_kind": lt["kl_kind"], "kl_coef": lt["kl_coef"], "ref": ref, "ent_coef": lt["ent_coef"]}


def oracle_token_weights(wl, lt):
    """Per-token gradient scales of the oracle's timed sample: the oracle's own dL/dl_t of the
    aggregation mode (oracle.aggregate.token_scale), the workload's rows taken as one step."""
    from oracle import aggregate as OG
    return OG.token_scale(wl.tok_off, wl.mask, OG.TOKEN_MEAN if lt is None else lt["agg"])


def oracle_lmhead_rate(wl, n_tokens: int, budget_s: float, lt=None):
    """Time the float64 LM-head oracle (z = h W^T, the objective, d_h and dW; the regularisers
    of ``lt`` when given) on `n_tokens` hidden states of a host-drawn sample at the workload's
    V and H, repeating the call until `budget_s` has passed (at least once). Returns (valid
    tokens/s, tokens timed, seconds)."""
    from oracle import loss as OL
    from rl_post_token_gb300 import workloads as W

    H = wl.extra["H"]
    n = min(wl.T, n_tokens)
    rng = np.random.default_rng(wl.seed + 7)
    h = W.bf16_round_bits(rng.standard_normal((n, H), dtype=np.float32) * np.float32(wl.extra["h_std"]))
    w = W.bf16_round_bits(rng.standard_normal((wl.V, H), dtype=np.float32) * np.float32(wl.extra["w_std"]))
    tgt, msk, adv = wl.target[:n], wl.mask[:n], np.where(np.arange(n) % 2, 1.0, -1.0)
    terms = oracle_terms(lt, np.random.default_rng(wl.seed + 1).normal(-10.0, 0.1, n))
    scale = oracle_token_weights(wl, lt)[:n]
    done, t0 = 0, time.perf_counter()
    while True:
        OL.lmhead_fwd_bwd(h, w, tgt, None, adv, msk, wl.eps, scale, terms=terms)
        done += int(msk.sum())
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return done / dt, done, dt


def _blas_threads() -> int:
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(k, "")
        if v.isdigit() and int(v) > 0:
            return int(v)
    return os.cpu_count() or 1


def lmhead_config(wl) -> dict:
    """The `config` of an LM-head line: the same dict in the library arm and the reference arm."""
    T, V, Hd = wl.T, wl.V, wl.extra["H"]
    return {"workload": WORKLOAD_TEXT["lmhead"], "tokens": int(T), "vocab": int(V), "hidden": int(Hd),
            "backward": "logits recomputed per vocabulary chunk (%d chunks), no [T, V] matrix stored"
                        % lmhead_chunks(V),
            "l2": "weights 622 MB + hidden 64 MB read per step, larger than L2; no flush"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import planner as OP
    from rl_post_token_gb300 import workloads as W
    ov = {"rows": args.rows} if args.rows else {}
    if args.rows and args.workload == "qwen_step":
        ov.update(mini=args.rows, micro=args.rows)
    if args.workload == "lmhead" and args.lm_tokens:
        ov = {"tokens": args.lm_tokens}
    wl = W.make_workload(args.workload, seed=0, **ov)
    lt = cli_terms(args)
    if args.workload == "lmhead":
        config = dict(lmhead_config(wl), **({"terms": lt["text"]} if lt["text"] else {}))
    else:
        # the same config as the library arm's line; the exec rows from the oracle's planner
        pl = OP.plan(OP.PlanConfig(**wl.plan), wl.row_len, wl.row_valid, seg_counts=wl.seg_counts)
        exec_tokens = int(sum(int(wl.row_len[j]) for j in pl.row_src))
        config = workload_config(args, wl, exec_tokens, world, args.workload, lt["text"])
    per_step_s = 0.5
    if args.workload == "lmhead":
        # one call of the LM-head oracle on 4 tokens per step (its products use every BLAS thread)
        rate = lambda budget: oracle_lmhead_rate(wl, 4, budget, lt)
        cores = _blas_threads()
        sample = "float64 numpy LM-head oracle (z = h W^T, objective, d_h, dW), 4 host-drawn tokens per step"
    else:
        rate = lambda budget: oracle_sample_rate(wl, 16, budget, lt)
        cores = 1
        sample = (f"float64 numpy oracle, first 16 tokens of a host-drawn batch of the workload, "
                  f"{per_step_s}s per step")
    for _ in range(args.warmup):
        rate(per_step_s / 4)
    done, dt = 0, 0.0
    for _ in range(args.steps):
        _, n, d = rate(per_step_s)
        done += n
        dt += d
    v = done / dt
    line = {
        "impl": "reference", "metric": LMHEAD_METRIC if args.workload == "lmhead" else METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "host_cpus": os.cpu_count(), "kind": "oracle",
                         "sample": sample + (" (rank 0 only)" if world > 1 else "")},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---- the library arm ------------------------------------------------------------------------------

class Batch:
    """Device-resident inputs and outputs of one collected batch."""

    def __init__(self, wl, device, kl_kind=0, kl_coef=0.0, ent_coef=0.0, agg=0):
        import torch
        from rl_post_token_gb300 import _lib
        from rl_post_token_gb300 import step as S
        from rl_post_token_gb300 import workloads as W

        self.wl = wl
        self.dev = device
        # a step's chunks alternate between the caller's stream and this one (None: one stream)
        self.side = None if os.environ.get("GRPO_ONE_STREAM") == "1" else torch.cuda.Stream(device)
        # each optimizer step's finish on its own stream, beside the next step's chunks
        self.fin = None if self.side is None else torch.cuda.Stream(device)
        self.bp = S.plan_batch(wl.plan, wl.row_len, wl.row_valid, wl.seg_counts)
        Te = self.bp.exec_tokens
        T = wl.T
        self.logits = W.make_logits(wl, device, rows=Te)       # exec order, as a model emits
        self.dlogits = torch.empty_like(self.logits)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        self.target, self.mask, self.rewards = t(wl.target), t(wl.mask), t(wl.rewards)
        self.row_tok_off = t(wl.tok_off)
        self.row_rollout = t(wl.row_rollout)
        self.tok_src = None if self.bp.tok_src is None else t(self.bp.tok_src)
        self.tok_src_host = None
        if self.tok_src is not None:  # pinned double buffer for the per-step plan upload
            self.tok_src_host = [torch.empty(self.tok_src.numel(), dtype=torch.int64, pin_memory=True)
                                 for _ in range(2)]
            self.tok_src_free = [None, None]
        self.adv_rollout = torch.empty_like(self.rewards)
        self.adv_tok = torch.empty(T, dtype=torch.float32, device=device)
        self.loss_tok = torch.empty(T, dtype=torch.float32, device=device)
        self.logp_tok = torch.empty(T, dtype=torch.float32, device=device)
        self.accs = torch.zeros(self.bp.n_steps * _lib.ACC_BYTES, dtype=torch.uint8, device=device)
        # pi_old from the ahead pass (forward only, before any pi_old exists), plus seeded noise
        self.old = None
        self.run(with_grad=False)
        self.old = self.logp_tok + t(wl.old_noise)
        # regularisers of the training step (not of the pi_old pass): a reference policy's
        # log-probs drawn like pi_old's (the ahead pass's log-probs plus seeded noise), and the
        # per-token entropy as an output
        self.terms, self.ref = None, None
        if kl_kind or ent_coef:
            self.terms = {"kl_kind": kl_kind, "kl_coef": kl_coef, "ent_coef": ent_coef}
            if kl_kind:
                noise = np.random.default_rng(wl.seed + 1).normal(0.0, 0.1, T).astype(np.float32)
                self.ref = self.old - t(wl.old_noise) + t(noise)
                self.terms["ref_logp"] = self.ref
            if ent_coef:
                self.terms["entropy_tok"] = torch.empty(T, dtype=torch.float32, device=device)
        # the loss aggregation mode; seq-mean-token-mean needs the planner's per-token weights
        self.agg, self.w_tok = agg, None
        if agg == _lib.AGG_SEQ_MEAN_TOKEN_MEAN:
            self.w_tok = t(self.bp.token_weights(agg)[1])
        torch.cuda.synchronize(device)
        self.n_step = 0

    def replan(self, stream):
        """The host planner runs every step; its token index goes up through pinned memory."""
        import torch
        from rl_post_token_gb300 import step as S
        wl = self.wl
        self.bp = S.plan_batch(wl.plan, wl.row_len, wl.row_valid, wl.seg_counts)
        if self.tok_src is not None:
            k = self.n_step % 2
            if self.tok_src_free[k] is not None:
                self.tok_src_free[k].synchronize()
            self.tok_src_host[k].numpy()[:] = self.bp.tok_src
            self.tok_src.copy_(self.tok_src_host[k], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(stream)
            self.tok_src_free[k] = ev
        self.n_step += 1

    def run(self, with_grad=True, stream=None, chunk_ready=None, launch_events=None, logits_host=None,
            staging=None, copy_stream=None, block_rows=1024):
        from rl_post_token_gb300 import _lib
        from rl_post_token_gb300 import step as S
        host = logits_host is not None
        return S.run_batch(self.bp, side_stream=None if host else self.side, logits=None if host else self.logits,
                           finish_stream=None if host else self.fin,
                           logits_host=logits_host, staging=staging, copy_stream=copy_stream, block_rows=block_rows,
                           dlogits=self.dlogits if with_grad else None,
                           target=self.target, old_logp=self.old, mask=self.mask, adv_tok=self.adv_tok,
                           loss_tok=self.loss_tok, logp_tok=self.logp_tok, accs=self.accs,
                           clip_eps=self.wl.eps, rewards=self.rewards, adv_rollout=self.adv_rollout,
                           group_size=self.wl.group_size, row_tok_off=self.row_tok_off,
                           row_rollout=self.row_rollout, tok_src=self.tok_src, V=self.wl.V,
                           stream=stream, chunk_ready=chunk_ready, launch_events=launch_events,
                           terms=self.terms if with_grad else None,
                           agg=self.agg if with_grad else _lib.AGG_TOKEN_MEAN,
                           w_tok=self.w_tok if with_grad else None)

    def algorithmic_bytes(self):
        """Bytes the method must move per batch in the row pass: a valid token reads its logits
        row and writes its dlogits row plus its side inputs and outputs (target, pi_old,
        advantage, mask, loss, log-prob, and the token index when the order is permuted); a
        masked or padding token writes a zero row."""
        wl = self.wl
        rowb = wl.V * wl.elem_bytes
        idx = 8 if self.tok_src is not None else 0
        extra = 0  # the terms' per-token inputs (reference log-prob, aggregation weight), output (entropy)
        if self.terms is not None:
            extra = (4 if self.terms.get("ref_logp") is not None else 0) + \
                    (4 if self.terms.get("entropy_tok") is not None else 0)
        if self.w_tok is not None:
            extra += 4
        valid = wl.n_valid  # each valid input token runs exactly once; padding rows are masked
        masked = self.bp.exec_tokens - valid
        return valid * (2 * rowb + 4 + 4 + 4 + 1 + 4 + 4 + idx + extra) + masked * (rowb + 1 + idx)


def cli_terms(args) -> dict:
    """The regularisers and aggregation mode that the command line asks for (--kl, --kl-coef,
    --ent-coef, --agg), with their text for the line's config."""
    from rl_post_token_gb300 import _lib
    kl = getattr(args, "kl", "none")
    agg_name = getattr(args, "agg", "token-mean")
    out = {"kl_kind": {"none": 0, "k1": _lib.KL_K1, "k3": _lib.KL_K3}[kl],
           "kl_coef": float(getattr(args, "kl_coef", 0.0)), "ent_coef": float(getattr(args, "ent_coef", 0.0)),
           "agg": {"token-mean": _lib.AGG_TOKEN_MEAN, "seq-mean-token-sum": _lib.AGG_SEQ_MEAN_TOKEN_SUM,
                   "seq-mean-token-mean": _lib.AGG_SEQ_MEAN_TOKEN_MEAN}[agg_name]}
    out["text"] = ", ".join(([f"KL {kl} coef {out['kl_coef']}"] if out["kl_kind"] else []) +
                            ([f"entropy bonus coef {out['ent_coef']} (entropy written per token)"]
                             if out["ent_coef"] else []) +
                            ([f"aggregation {agg_name}"] if out["agg"] != _lib.AGG_TOKEN_MEAN else []))
    return out


def lmhead_chunks(V):
    """Vocabulary chunks of the LM-head backward: ceil(V/256) tiles in chunks of at most 66."""
    tiles = -(-V // 256)
    return -(-tiles // 66)


def run_lmhead(args):
    """The fused LM-head workload as the line's headline (one GPU only)."""
    import torch

    rank, world, local = dist_env()
    if world > 1:
        raise SystemExit("--workload lmhead runs on one GPU only")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from rl_post_token_gb300 import build as B
    B.build()
    line = measure_lmhead(args, device, rank, local)
    line.update({"n_gpus": 1, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                 "data": "synthetic"})
    print(json.dumps(line), flush=True)
    return 0


def measure_lmhead(args, device, rank=0, local=0, with_e2e=True, with_cpu=True):
    """Fused LM-head step: advantage, one grpo_lmhead_loss_fwd_bwd call (forward, dlogits, d_h
    and dW, no [T, V] matrix stored: the backward recomputes each vocabulary chunk's logits for
    the tokens with a nonzero gradient), the finish. Roofline: tensor, 2*N*V*H + 4*T_live*V*H
    algorithmic flops (the forward GEMM over the N valid tokens, the two backward GEMMs over
    the live ones; the recompute's 2*T_live*V*H is not credited) over the LM-head call's time,
    timed with CUDA events around each call on its stream. --lm-mask-frac masks a share of the
    tokens and --lm-skip-masked sets GRPO_LMHEAD_SKIP_MASKED."""
    import torch
    from rl_post_token_gb300 import _lib
    from rl_post_token_gb300 import workloads as W

    _lib.lib()
    wl = W.make_workload("lmhead", seed=rank, **({"tokens": args.lm_tokens} if args.lm_tokens else {}))
    mask_frac = float(getattr(args, "lm_mask_frac", 0.0))
    skip_masked = bool(getattr(args, "lm_skip_masked", False))
    if mask_frac > 0:  # a seeded share of the tokens masked (padding), for the masked-token flag
        wl.mask[np.random.default_rng(wl.seed + 5).random(wl.T) < mask_frac] = 0
    T, V, Hd = wl.T, wl.V, wl.extra["H"]
    h, Wt = W.make_lmhead_inputs(wl, device)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    target, mask, rewards = t(wl.target), t(wl.mask), t(wl.rewards)
    adv_r = torch.empty_like(rewards)
    adv = torch.empty(T, device=device)
    row_tok_off, row_rollout = t(wl.tok_off), t(wl.row_rollout)
    d_h = torch.empty((T, Hd), device=device)
    dW = torch.empty((V, Hd), device=device)
    loss = torch.empty(T, device=device)
    logp = torch.empty(T, device=device)
    acc = _lib.new_step_acc(device)
    ws = torch.empty(_lib.grpo_lmhead_workspace_size(T, V, Hd), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    N = wl.n_valid
    call_evs = []
    # the training step's regularisers and loss aggregation, as for the row-pass workloads (the
    # pi_old pass takes neither); the aggregation's grad scale, weights and divisor come from
    # grpo_plan_token_weights over the step's rows
    lt = cli_terms(args)
    gs, divisor, w_tok = 1.0 / max(N, 1), -1, None
    if lt["agg"] != _lib.AGG_TOKEN_MEAN:
        div, w, sc = _lib.grpo_plan_token_weights({"n_steps": 1, "step_in_row_off": [0, len(wl.row_len)]},
                                                  wl.row_len, wl.row_valid, lt["agg"], want_scale=True)
        gs, divisor = float(sc[0]), int(div[0])
        w_tok = t(w) if lt["agg"] == _lib.AGG_SEQ_MEAN_TOKEN_MEAN else None
    terms = None

    def step(grads=True, old=None, w=ws, evs=None):
        _lib.grpo_group_advantage(rewards, wl.group_size, 1e-6, True, adv_r, row_rollout, row_tok_off, adv)
        if evs is not None:
            evs.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
            evs[-1][0].record(stream)
        tm = terms if grads else None
        _lib.grpo_lmhead_loss_fwd_bwd(h, Wt, target, old, adv, mask, wl.eps, gs if grads else 1.0 / max(N, 1),
                                      d_h if grads else None, dW if grads else None, loss, logp, acc, w, terms=tm,
                                      skip_masked=skip_masked)
        if evs is not None:
            evs[-1][1].record(stream)
        if grads and (w_tok is not None or divisor >= 0):
            _lib.grpo_finish_step_ex(acc, loss, w_tok=w_tok, divisor=divisor, expected_N=N, sync=False)
        else:
            _lib.grpo_finish_step(acc, loss, expected_N=N, sync=False)

    step(grads=False)  # pi_old by the ahead pass, then seeded noise
    old = logp + t(wl.old_noise)
    if lt["kl_kind"] or lt["ent_coef"] or w_tok is not None:
        terms = {"kl_kind": lt["kl_kind"], "kl_coef": lt["kl_coef"], "ent_coef": lt["ent_coef"], "w_tok": w_tok}
        if lt["kl_kind"]:  # a reference policy drawn like pi_old: the policy's log-probs plus noise
            noise = np.random.default_rng(wl.seed + 1).normal(0.0, 0.1, T).astype(np.float32)
            terms["ref_logp"] = logp + t(noise)
        if lt["ent_coef"]:
            terms["entropy_tok"] = torch.empty(T, dtype=torch.float32, device=device)
    torch.cuda.synchronize(device)
    # the clock sampler first, then the warm-up steps right before the timed ones (no idle gap
    # in which the power-capped GPU could recover before the timed region)
    clocks = ClockSampler(_gpu_index(local), os.path.join(args.clocks_dir, f"clocks_lmhead_rank{rank}.csv"))
    time.sleep(0.5)
    for _ in range(max(args.warmup, 3)):
        step(old=old)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step(old=old, evs=call_evs)
    e1.record(stream)
    torch.cuda.synchronize(device)
    full_s = e0.elapsed_time(e1) / 1e3 / args.steps
    call_s = sum(a.elapsed_time(b) for a, b in call_evs) / 1e3 / len(call_evs)
    res = _lib.read_step_result(acc)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        step(grads=False, old=old)
    f1.record(stream)
    torch.cuda.synchronize(device)
    fwd_s = f0.elapsed_time(f1) / 1e3 / args.steps
    clk = clocks.stop()

    # the e2e step: the same call on an input set that comes up from pinned host memory
    dev_in = {"h": h, "Wt": Wt, "target": target, "mask": mask, "rewards": rewards, "old": old}
    if terms is not None and terms.get("ref_logp") is not None:
        dev_in["ref"] = terms["ref_logp"]
    if w_tok is not None:
        dev_in["w_tok"] = w_tok

    def train_call(s):
        _lib.grpo_group_advantage(s["rewards"], wl.group_size, 1e-6, True, adv_r, row_rollout, row_tok_off, adv)
        tm = None if terms is None else dict(terms, ref_logp=s.get("ref"), w_tok=s.get("w_tok"))
        _lib.grpo_lmhead_loss_fwd_bwd(s["h"], s["Wt"], s["target"], s["old"], adv, s["mask"], wl.eps, gs,
                                      d_h, dW, loss, logp, acc, ws, terms=tm, skip_masked=skip_masked)
        if w_tok is not None or divisor >= 0:
            _lib.grpo_finish_step_ex(acc, loss, w_tok=s.get("w_tok"), divisor=divisor, expected_N=N, sync=False)
        else:
            _lib.grpo_finish_step(acc, loss, expected_N=N, sync=False)

    e2e = measure_lmhead_e2e(args, wl, device, stream, dev_in, train_call, acc, res) if with_e2e else None
    # the backward's live tokens (a nonzero dlogits row): with the KL term or the entropy bonus
    # every valid token; otherwise the valid tokens with a nonzero advantage that the clip did
    # not stop (a clipped token has a nonzero advantage by definition)
    if terms is not None and (terms["kl_kind"] or terms["ent_coef"]):
        t_live = N
    else:
        t_live = int(((adv != 0) & (mask != 0)).sum().item()) - int(res["n_clipped"])
    # credited: the forward over the valid tokens (every token in the bench's workload) and the
    # two backward products over the live ones (a dead token's products are exact zeros);
    # executed: the forward over every token (or the valid ones with the masked-token flag)
    # plus the live tokens' recompute
    flops = (2.0 * N + 4.0 * t_live) * V * Hd
    executed = (2.0 * (N if skip_masked else T) + 6.0 * t_live) * V * Hd
    peak, kind = bf16_peak(sustained=True)
    line = {
        "metric": LMHEAD_METRIC,
        "value": N / full_s, "unit": UNIT, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": 1e3 * full_s, "dtype": "bf16",
        "config": dict(lmhead_config(wl), **({"terms": lt["text"]} if lt["text"] else {}),
                       **({"masked_share": mask_frac} if mask_frac > 0 else {}),
                       **({"skip_masked": True} if skip_masked else {})),
        "workspace_gb": ws.numel() / 1e9,
        "roofline": {"bound": "tensor", "achieved": flops / call_s / 1e12, "peak": peak, "unit": "TFLOP/s",
                     "frac": flops / call_s / 1e12 / peak, "peak_source": f"{kind} bf16_tflops_sustained",
                     "kernel": "grpo_lmhead_loss_fwd_bwd (its GEMM launches and the per-token reduce), CUDA events "
                               "around each call",
                     "ms_per_call": 1e3 * call_s, "flops_per_call": flops,
                     "flops_what": "2*N*V*H (forward, the valid tokens) + 4*T_live*V*H (d_h and dW over the "
                                   "tokens with a nonzero dlogits row)",
                     "live_tokens": t_live, "dense_flops_per_call": 6.0 * T * V * Hd,
                     "executed_flops_per_call": executed,
                     "executed_tflops": executed / call_s / 1e12, "traffic": None},
        "forward_only": {"ms": 1e3 * fwd_s, "tflops": 2.0 * T * V * Hd / fwd_s / 1e12,
                         "what": "softmax-partials GEMM pass + per-token reduce (2*T*V*H flops)"},
        "step_result": {k: res[k] for k in ("loss", "n_valid", "clipfrac", "status")},
        # per step: the advantage (2), pass A and the per-token reduce (2), the live-token
        # partition and gather (2), per vocabulary chunk the dlogits recompute, the d_h and the
        # dW GEMM (3), the finish (1)
        "gpu_launches": (7 + 3 * lmhead_chunks(V)) * args.steps,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if clk is not None:
        line["clocks"] = clk
    if with_cpu and rank == 0 and not args.no_cpu_baseline:
        v, n, dt = oracle_lmhead_rate(wl, 16, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": _blas_threads(), "host_cpus": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"float64 numpy LM-head oracle (z = h W^T, objective, d_h, dW; its "
                                          f"products on every BLAS thread), 16 host-drawn tokens per call, "
                                          f"{n} valid tokens in {dt:.1f} s"}
    return line


def measure_lmhead_e2e(args, wl, device, stream, dev_in, train_call, acc, ref_res):
    """The LM-head step through the public API with every step's inputs (hidden states, weights,
    side arrays, the regularisers' per-token inputs) starting in pinned host memory: copied up
    on a copy stream into one of two device input sets, the next step's copy overlapping this
    step's compute (the first step's copy does not overlap); ``train_call(set)`` runs the
    step's calls on a set; the step result is read back every step."""
    import torch
    from rl_post_token_gb300 import _lib

    N = wl.n_valid
    host = {k: v.cpu().pin_memory() for k, v in dev_in.items()}
    sets = [dev_in, {k: torch.empty_like(v) for k, v in dev_in.items()}]
    host_res = torch.empty(64, dtype=torch.uint8, pin_memory=True)
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    copy = torch.cuda.Stream(device)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    used = [torch.cuda.Event(), torch.cuda.Event()]
    for e in used:
        e.record(stream)

    def upload(k):
        s = sets[k % 2]
        copy.wait_event(used[k % 2])  # the step that last read this set is done
        with torch.cuda.stream(copy):
            for name, v in host.items():
                s[name].copy_(v, non_blocking=True)
        copied[k % 2].record(copy)

    def e2e_step(k, n):
        if k == 0:
            upload(0)
        if k + 1 < n:
            upload(k + 1)
        s = sets[k % 2]
        stream.wait_event(copied[k % 2])
        train_call(s)
        used[k % 2].record(stream)
        host_res.copy_(acc[64:128], non_blocking=True)
        stream.synchronize()

    for k in range(3):  # warm-up steps, as for the device-timed region
        e2e_step(k, 3)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for k in range(e2e_steps):
        e2e_step(k, e2e_steps)
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    copy.synchronize()
    e2e_res = _lib.read_step_result(acc)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    keys = ("loss", "n_valid", "clipfrac", "status")
    return {"value": N / e2e_s, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(host_res.numel()), "steps": e2e_steps,
            "how": "hidden states, weights and side inputs copied from pinned host memory every step on a "
                   "copy stream into one of two device input sets (the next step's copy overlaps this step's "
                   "compute, the first step's does not), the step result read back every step",
            "step_result_matches": all(e2e_res[k] == ref_res[k] for k in keys)}


def time_rowpass(args, batch, device, stream, world, local, clocks_name):
    """Warm up, then time `args.steps` whole batches between a barrier and a synchronize on
    both sides, sampling the clocks during the timed region. Returns the timing record."""
    import torch
    from rl_post_token_gb300 import step as S

    # the clock sampler starts first (it takes a moment to come up), then the warm-up steps run
    # right before the timed ones, so the GPU does not idle between the two
    clocks = ClockSampler(_gpu_index(local), os.path.join(args.clocks_dir, clocks_name))
    time.sleep(0.5)
    for _ in range(max(args.warmup, 3)):
        batch.replan(stream)
        batch.run(stream=stream)
    barrier(world, device)
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    evs = []
    start.record(stream)
    for _ in range(args.steps):
        batch.replan(stream)
        launches += batch.run(stream=stream, launch_events=evs)
    end.record(stream)
    torch.cuda.synchronize(device)
    barrier(world, device)
    clk = clocks.stop()
    elapsed = start.elapsed_time(end) / 1e3
    # the dominant kernel: row-pass launches timed on the streams they run on inside the timed
    # region (the union of their intervals: a step's chunks alternate between two streams)
    row_s = busy_seconds(start, evs)
    per_launch_bytes = batch.algorithmic_bytes() / (len(evs) / args.steps)
    return {"elapsed": elapsed, "launches": launches, "n_launches": len(evs), "row_s": row_s, "clocks": clk,
            "achieved_gbs": per_launch_bytes / (row_s / len(evs)) / 1e9,
            "results": S.read_results(batch.accs, batch.bp.n_steps)}


def workload_config(args, wl, exec_tokens: int, world: int, workload: str, terms_text: str = "") -> dict:
    """The `config` of a row-pass line: the same dict in the library arm and the reference arm."""
    return {"workload": WORKLOAD_TEXT[workload] + (f" [rows overridden: {args.rows}]" if args.rows else "")
                        + (f" [loss terms: {terms_text}]" if terms_text else ""),
            "valid_tokens_per_step": int(wl.n_valid),
            "logits_rows_per_step": int(exec_tokens), "vocab": int(wl.V),
            "l2": "inputs larger than L2 (%.1f GB of logits per step), no flush"
                  % (exec_tokens * wl.V * wl.elem_bytes / 1e9),
            "parallelism": f"{world} independent replicas" if world > 1 else "1 GPU"}


def rowpass_entry(args, wl, batch, tm, world, device, workload, traffic_per_valid=None, terms_text=""):
    """The JSON record of one row-pass workload: whole-job valid tokens/s, the row pass's
    roofline (algorithmic bytes per launch over its average launch time), clocks, results."""
    units = wl.n_valid * args.steps
    max_el, all_units = reduce_timing(tm["elapsed"], units, world, device)
    peak, peak_kind = hbm_peak()
    launches_per_step = tm["n_launches"] / args.steps
    entry = {
        "metric": METRIC, "value": all_units / max_el, "unit": UNIT, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": 1e3 * max_el / args.steps,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "config": workload_config(args, wl, batch.bp.exec_tokens, world, workload, terms_text),
        "roofline": {"bound": "hbm", "achieved": tm["achieved_gbs"], "peak": peak, "unit": "GB/s",
                     "frac": tm["achieved_gbs"] / peak, "peak_source": f"{peak_kind} hbm_gbs",
                     "frac_of_8tbs": tm["achieved_gbs"] / 8000.0,
                     "kernel": "row pass (grpo_logprob_loss_fwd_bwd" + (f"_ex: {terms_text})" if terms_text else ")"),
                     "row_pass_share_of_step": tm["row_s"] / tm["elapsed"],
                     "traffic": None if traffic_per_valid is None else traffic_per_valid * wl.n_valid / launches_per_step},
        "gpu_launches": tm["launches"],
        "step_results": [{k: r[k] for k in ("loss", "n_valid", "clipfrac", "status")} for r in tm["results"]],
    }
    if tm["clocks"] is not None:
        entry["clocks"] = tm["clocks"]
    return entry


def run_gb300(args):
    import torch

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    from rl_post_token_gb300 import build as B
    if rank == 0:
        B.build()
    barrier(world, device)
    from rl_post_token_gb300 import _lib
    from rl_post_token_gb300 import workloads as W

    _lib.lib()
    ov = {"rows": args.rows} if args.rows else {}
    if args.rows and args.workload == "qwen_step":
        ov.update(mini=args.rows, micro=args.rows)
    wl = W.make_workload(args.workload, seed=rank, **ov)
    lt = cli_terms(args)
    batch = Batch(wl, device, kl_kind=lt["kl_kind"], kl_coef=lt["kl_coef"], ent_coef=lt["ent_coef"], agg=lt["agg"])
    terms_text = lt["text"]
    stream = torch.cuda.current_stream(device)
    tm = time_rowpass(args, batch, device, stream, world, local, f"clocks_rank{rank}.csv")
    # the committed capture is of the default workload's instance without terms
    tpv = profiled_traffic() if args.workload == "qwen_step" and not terms_text and not args.rows else None
    line = rowpass_entry(args, wl, batch, tm, world, device, args.workload, tpv, terms_text)
    line.update({"n_gpus": world, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                 "data": "synthetic"})

    ahead = run_ahead(batch, stream, steps=min(args.steps, 30))
    barrier(world, device)
    e2e = run_e2e(batch, device, stream, steps=min(args.steps, args.e2e_steps), ref_results=tm["results"])
    # whole job: every rank's tokens over the slowest rank's time, as for `value`
    e2e_el, e2e_units = reduce_timing(e2e.pop("elapsed_s"), e2e.pop("units"), world, device)
    e2e["value"] = e2e_units / e2e_el
    line["e2e"] = e2e
    # a read-only stream: the measured copy figure (reads and writes) is not its ceiling, so the
    # fraction of the nominal 8 TB/s is given beside it
    line["ahead_pass"] = dict(ahead, frac=ahead["achieved_gbs"] / hbm_peak()[0],
                              frac_of_8tbs=ahead["achieved_gbs"] / 8000.0, per_gpu=True)
    if rank == 0 and not args.no_cpu_baseline:
        v, n, dt = oracle_sample_rate(wl, 16, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "host_cpus": os.cpu_count(), "kind": "oracle",
                                "sample": f"float64 numpy oracle (one thread) on {n} valid tokens "
                                          f"({dt:.1f} s) of a host-drawn sample of the workload"}
    del batch

    # the other workloads of the method, timed the same way on the same GPU (one GPU only)
    if world == 1 and args.workload == "qwen_step" and not args.no_extra_workloads and not args.rows \
            and not terms_text:
        extra = {}
        for name in ("dynamic", "compaction"):
            torch.cuda.empty_cache()
            wx = W.make_workload(name, seed=rank)
            bx = Batch(wx, device)
            tmx = time_rowpass(args, bx, device, stream, world, local, f"clocks_{name}_rank{rank}.csv")
            extra[name] = rowpass_entry(args, wx, bx, tmx, world, device, name)
            del bx
        # the headline step with the regularisers: KL k3 to a reference policy and the entropy
        # bonus (the entropy written per token)
        torch.cuda.empty_cache()
        wx = W.make_workload("qwen_step", seed=rank)
        bx = Batch(wx, device, kl_kind=_lib.KL_K3, kl_coef=0.05, ent_coef=0.01)
        tmx = time_rowpass(args, bx, device, stream, world, local, f"clocks_terms_rank{rank}.csv")
        extra["qwen_step_kl3_entropy"] = rowpass_entry(args, wx, bx, tmx, world, device, "qwen_step", None,
                                                       "KL k3 coef 0.05, entropy bonus coef 0.01 (entropy "
                                                       "written per token)")
        del bx
        torch.cuda.empty_cache()
        extra["lmhead"] = measure_lmhead(args, device, rank, local, with_e2e=False, with_cpu=False)
        # the same step with the KL term to a reference policy: every token has a gradient, so
        # the backward runs over all of them (the dense case beside the plain step's live ones)
        torch.cuda.empty_cache()
        extra["lmhead_kl3"] = measure_lmhead(argparse.Namespace(**dict(vars(args), kl="k3", kl_coef=0.05)), device,
                                             rank, local, with_e2e=False, with_cpu=False)
        line["workloads"] = extra
        line["gpu_launches"] += sum(e["gpu_launches"] for e in extra.values())
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def busy_seconds(ref, evs):
    """Length of the union of the [start, end] intervals of event pairs (seconds), measured from
    the reference event: the time some row-pass launch was running. With a step's chunks on
    two streams the launches overlap at their ends, so their durations must not be summed."""
    iv = sorted((ref.elapsed_time(a), ref.elapsed_time(b)) for a, b in evs)
    total, cur_a, cur_b = 0.0, None, None
    for a, b in iv:
        if cur_b is None or a > cur_b:
            if cur_b is not None:
                total += cur_b - cur_a
            cur_a, cur_b = a, b
        else:
            cur_b = max(cur_b, b)
    if cur_b is not None:
        total += cur_b - cur_a
    return total / 1e3


def run_ahead(batch, stream, steps: int):
    """The pi_old ahead pass: the same batch forward only (no dlogits), timed with CUDA events
    around each row-pass launch. Algorithmic bytes: each valid token reads its logits row and
    its side inputs and writes its log-prob and loss."""
    import torch
    evs = []
    for _ in range(3):
        batch.run(with_grad=False, stream=stream)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        batch.run(with_grad=False, stream=stream, launch_events=evs)
    end.record(stream)
    torch.cuda.synchronize()
    wl = batch.wl
    row_s = busy_seconds(start, evs)
    idx = 8 if batch.tok_src is not None else 0
    per_batch = wl.n_valid * (wl.V * wl.elem_bytes + 4 + 4 + 4 + 1 + 4 + 4 + idx)
    return {"value": wl.n_valid * steps / (start.elapsed_time(end) / 1e3), "unit": UNIT,
            "achieved_gbs": per_batch * steps / row_s / 1e9, "steps": steps,
            "what": "forward-only row pass (pi_old ahead pass): log-prob and loss, no dlogits"}


def _gpu_index(local: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p for p in vis.split(",") if p.strip()]
    if parts and all(p.strip().isdigit() for p in parts) and local < len(parts):
        return int(parts[local])
    return local


# ---- host memory placement (NUMA) -----------------------------------------------------------------

def gpu_numa_node(local: int):
    """NUMA node the GPU's PCI function reports (sysfs numa_node), or None if unknown."""
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader",
                              "-i", str(_gpu_index(local))], capture_output=True, text=True, timeout=20).stdout
        bus = out.strip().splitlines()[0].strip().lower()
        dom, rest = bus.split(":", 1)
        path = f"/sys/bus/pci/devices/{int(dom, 16):04x}:{rest}/numa_node"
        node = int(open(path).read().strip())
        return node if node >= 0 else None
    except Exception:
        return None


def node_cpus(node: int):
    """CPUs of a NUMA node (sysfs cpulist), or an empty set."""
    cpus = set()
    try:
        for part in open(f"/sys/devices/system/node/node{node}/cpulist").read().strip().split(","):
            if "-" in part:
                a, b = part.split("-")
                cpus.update(range(int(a), int(b) + 1))
            elif part:
                cpus.add(int(part))
    except OSError:
        pass
    return cpus


def page_nodes(t, samples: int = 16):
    """NUMA nodes of `samples` pages spread over a host tensor (move_pages with no target
    nodes only reports where each page is), as {node: pages}; None if the query fails."""
    import ctypes
    import platform

    nr = {"aarch64": 239, "x86_64": 279}.get(platform.machine())
    if nr is None or t.numel() == 0:
        return None
    base, nbytes = t.data_ptr(), t.numel() * t.element_size()
    page = os.sysconf("SC_PAGE_SIZE")
    addrs = sorted({(base + k * nbytes // samples) // page * page for k in range(samples)})
    n = len(addrs)
    pages = (ctypes.c_void_p * n)(*addrs)
    status = (ctypes.c_int * n)()
    libc = ctypes.CDLL(None, use_errno=True)
    libc.syscall.restype = ctypes.c_long
    rc = libc.syscall(ctypes.c_long(nr), ctypes.c_int(0), ctypes.c_ulong(n), pages, None, status, ctypes.c_int(0))
    if rc != 0:
        return None
    out = {}
    for v in status:
        out[int(v)] = out.get(int(v), 0) + 1
    return out


def pinned_like(t, local: int):
    """A pinned host copy of device tensor `t`, allocated (and first touched) by this thread
    while it is bound to the CPUs of the GPU's NUMA node, so that its pages sit on that node.
    Returns (tensor, placement record)."""
    import torch

    node = gpu_numa_node(local)
    cpus = node_cpus(node) if node is not None else set()
    old = os.sched_getaffinity(0)
    bound = False
    if cpus and (cpus & old):
        os.sched_setaffinity(0, cpus & old)
        bound = True
    try:
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.view(torch.uint8).zero_()  # first touch on the bound CPUs
    finally:
        if bound:
            os.sched_setaffinity(0, old)
    h.copy_(t)
    return h, {"gpu_numa_node": node, "bound_to_gpu_node": bound, "host_pages_by_node": page_nodes(h)}


def _d2h_copy_gbs(host, dev, stream, reps: int = 8) -> float:
    """GB/s of `reps` plain device->host copies into the start of the pinned tensor `host`."""
    import torch

    dst = host.reshape(-1).view(torch.uint8)
    n = min(dst.numel(), dev.numel())
    dst, dev = dst[:n], dev[:n]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        dst.copy_(dev, non_blocking=True)
        e0.record(stream)
        for _ in range(reps):
            dst.copy_(dev, non_blocking=True)
        e1.record(stream)
    stream.synchronize()
    return reps * n / (e0.elapsed_time(e1) / 1e3) / 1e9


def _h2d_copy_gbs(host, dev, stream, reps: int = 8) -> float:
    """GB/s of `reps` plain host->device copies from the start of the pinned tensor `host`
    into `dev` (`dev`'s size, or all of `host` if smaller), timed with CUDA events on
    `stream`: the host link's rate at that moment."""
    import torch

    src = host.reshape(-1).view(torch.uint8)
    n = min(src.numel(), dev.numel())
    src, dev = src[:n], dev[:n]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        dev.copy_(src, non_blocking=True)
        e0.record(stream)
        for _ in range(reps):
            dev.copy_(src, non_blocking=True)
        e1.record(stream)
    stream.synchronize()
    return reps * dev.numel() / (e0.elapsed_time(e1) / 1e3) / 1e9


def run_e2e(batch, device, stream, steps: int, ref_results=None):
    """Same metric through the public API with HOST inputs. Every step:
    - the logits stream from pinned host memory through the library's host entry point
      (`grpo_logprob_loss_fwd_bwd_host`): 1024-row blocks into a two-block device staging
      buffer, the copies on a copy stream, each block's row pass waiting only for its own copy;
    - the side inputs are copied up;
    - the batch runs;
    - the step results are read back."""
    import torch

    host_logits, placement = pinned_like(batch.logits, device.index)
    side = {k: getattr(batch, k).cpu().pin_memory() for k in ("target", "mask", "rewards", "old")
            + (("ref",) if batch.ref is not None else ()) + (("w_tok",) if batch.w_tok is not None else ())}
    host_res = torch.empty(batch.accs.numel(), dtype=torch.uint8, pin_memory=True)
    block = 1024
    staging = torch.empty(2 * block * host_logits.stride(0) * host_logits.element_size(), dtype=torch.uint8,
                          device=device)
    copy = torch.cuda.Stream(device)
    torch.cuda.synchronize(device)

    def one_step():
        batch.replan(stream)
        with torch.cuda.stream(stream):
            for k, v in side.items():
                getattr(batch, k).copy_(v, non_blocking=True)
        batch.run(stream=stream, logits_host=host_logits, staging=staging, copy_stream=copy, block_rows=block)
        with torch.cuda.stream(stream):
            host_res.copy_(batch.accs, non_blocking=True)
        stream.synchronize()

    for _ in range(3):  # warm-up steps, as for the device-timed region
        one_step()
    link_before = _h2d_copy_gbs(host_logits, staging, copy)
    step_s = []
    t0 = time.perf_counter()
    for _ in range(steps):
        ts = time.perf_counter()
        one_step()
        step_s.append(time.perf_counter() - ts)
    dt = time.perf_counter() - t0
    link_after = _h2d_copy_gbs(host_logits, staging, copy)
    d2h_link = _d2h_copy_gbs(host_logits, staging, copy)
    from rl_post_token_gb300 import step as S
    keys = ("loss", "n_valid", "clipfrac", "status")
    got = [{k: r[k] for k in keys} for r in S.read_results(host_res, batch.bp.n_steps)]
    match = None if ref_results is None else got == [{k: r[k] for k in keys} for r in ref_results]
    h2d = host_logits.numel() * host_logits.element_size() + sum(v.numel() * v.element_size() for v in side.values())
    return {"value": batch.wl.n_valid * steps / dt, "elapsed_s": dt, "units": batch.wl.n_valid * steps,
            "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(host_res.numel()), "steps": steps,
            "h2d_gbs": h2d * steps / dt / 1e9,
            "step_ms": [round(1e3 * x, 2) for x in step_s],
            "value_at_median_step": batch.wl.n_valid / float(np.median(step_s)),
            "step_results_match": match,
            "link_copy_gbs": {"before": link_before, "after": link_after, "d2h": d2h_link,
                              "what": "plain pinned host->device copies of the staging buffer's size, "
                                      "on the copy stream, just before and just after the timed steps; "
                                      "d2h: device->host copies of the same size after them"},
            "host_placement": placement,
            "how": "pinned host logits streamed by grpo_logprob_loss_fwd_bwd_host (1024-row blocks through a "
                   "two-block device staging buffer, copies overlapped with the row pass); side inputs copied "
                   "and step results read back every step"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="qwen_step", choices=list(WORKLOAD_TEXT))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-dir", default=tempfile.gettempdir(),
                    help="where the raw clock samples of the timed region are written (CSV)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="time only the chosen workload (the default line also times the dynamic, compaction "
                         "and fused LM-head workloads)")
    ap.add_argument("--lm-tokens", type=int, default=0,
                    help="override the fused LM-head token count (smaller cases for profiling)")
    ap.add_argument("--lm-mask-frac", type=float, default=0.0,
                    help="mask a seeded share of the LM-head workload's tokens (padding)")
    ap.add_argument("--lm-skip-masked", action="store_true",
                    help="run the LM-head forward GEMM over the mask=1 tokens only (GRPO_LMHEAD_SKIP_MASKED)")
    ap.add_argument("--rows", type=int, default=0,
                    help="override the workload's row count (smaller cases for profiling)")
    ap.add_argument("--kl", default="none", choices=["none", "k1", "k3"],
                    help="add a KL term to a reference policy to the training step's loss")
    ap.add_argument("--kl-coef", type=float, default=0.05)
    ap.add_argument("--ent-coef", type=float, default=0.0,
                    help="add an entropy bonus (and the per-token entropy output) to the step's loss")
    ap.add_argument("--agg", default="token-mean", choices=["token-mean", "seq-mean-token-sum", "seq-mean-token-mean"],
                    help="the loss aggregation mode of the step")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "lmhead":
        return run_lmhead(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
