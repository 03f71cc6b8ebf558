"""Driver loop of one collected batch over the C-ABI entry points.

Host control flow only ("Sizing mini-batches and micro-batches", "The loop at a glance"):
plan -> group advantage -> for each optimizer step, for each chunk, the loss forward+backward
-> the step finish. Every piece of arithmetic runs in ``libgrpo.so``.

Layouts:
* per-token side inputs (target, mask, pi_old, advantage) and per-token outputs (loss_tok,
  logp_tok) are in INPUT order (rows in the order collected, tokens of a row consecutive);
* logits and dlogits are in EXEC order (the plan's rows, which is what a model produces
  chunk by chunk); ``tok_src`` maps exec tokens to input tokens and is None when the two
  orders coincide (fixed chunks).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import numpy as np

from . import _lib


@dataclass
class BatchPlan:
    plan: dict                      # grpo_plan_microbatches output
    row_tok_off: np.ndarray         # int64 [rows + 1], input order
    exec_tok_off: np.ndarray        # int64 [chunks + 1], exec order
    tok_src: Optional[np.ndarray]   # int64 [exec tokens] or None (identity)
    step_tok_range: List[tuple]     # input-order token range of each optimizer step
    step_exec_range: List[tuple]    # exec-order token range of each optimizer step
    row_len: np.ndarray             # int64 [rows], input order
    row_valid: np.ndarray           # int32 [rows], input order

    def token_weights(self, agg: int, want_w: bool = True):
        """(divisor per step, per-token weights float32 in input order or None) of a loss
        aggregation mode (``_lib.AGG_*``), from grpo_plan_token_weights."""
        return _lib.grpo_plan_token_weights(self.plan, self.row_len, self.row_valid, agg, want_w)

    @property
    def n_steps(self) -> int:
        return int(self.plan["n_steps"])

    @property
    def exec_tokens(self) -> int:
        return int(self.exec_tok_off[-1])


def plan_batch(cfg: dict, row_len, row_valid, seg_counts=None) -> BatchPlan:
    p = _lib.grpo_plan_microbatches(cfg, row_len, row_valid, seg_counts)
    rl = np.asarray(row_len, np.int64)
    row_tok_off = np.zeros(rl.shape[0] + 1, np.int64)
    np.cumsum(rl, out=row_tok_off[1:])
    exec_tok_off = np.zeros(p["n_chunks"] + 1, np.int64)
    np.cumsum(p["chunk_tokens"], out=exec_tok_off[1:])
    identity = p["n_rows"] == rl.shape[0] and np.array_equal(p["row_src"], np.arange(rl.shape[0]))
    tok_src = None if identity else _lib.grpo_plan_token_index(p, rl)
    steps, execs = [], []
    for s in range(p["n_steps"]):
        r0, r1 = p["step_in_row_off"][s], p["step_in_row_off"][s + 1]
        steps.append((int(row_tok_off[r0]), int(row_tok_off[r1])))
        c0, c1 = p["step_chunk_off"][s], p["step_chunk_off"][s + 1]
        execs.append((int(exec_tok_off[c0]), int(exec_tok_off[c1])))
    return BatchPlan(p, row_tok_off, exec_tok_off, tok_src, steps, execs, rl,
                     np.asarray(row_valid, np.int32))


def run_batch(bp: BatchPlan, *, logits, dlogits, target, old_logp, mask, adv_tok, loss_tok,
              logp_tok, accs, clip_eps: float, rewards=None, adv_rollout=None, group_size: int = 1,
              adv_eps: float = 1e-6, row_tok_off=None, row_rollout=None, tok_src=None,
              deferred: bool = False, V: Optional[int] = None, stream=None,
              chunk_ready=None, launch_events=None, agg: int = _lib.AGG_TOKEN_MEAN,
              w_tok=None, side_stream=None, terms: Optional[dict] = None, logits_host=None,
              staging=None, block_rows: int = 1024, copy_stream=None, finish_stream=None) -> int:
    """Enqueue the whole batch; returns the number of library kernel launches.

    ``accs`` is a uint8 device tensor of n_steps * 128 bytes (one accumulator per optimizer
    step, results read later with ``read_results``). If ``rewards`` is given the advantage is
    computed into ``adv_rollout``/``adv_tok`` first. ``chunk_ready[c]`` (optional CUDA event)
    is waited on before chunk c is launched, e.g. the end of its host-to-device copy;
    ``launch_events`` (optional list) receives a (start, end) event pair per row-pass launch.
    ``agg`` selects the loss aggregation mode; SEQ_MEAN_TOKEN_MEAN also needs ``w_tok``, the
    device copy of ``bp.token_weights(agg)[1]`` (input order).

    ``terms`` (optional): the regularisers every chunk's call adds, as for
    ``_lib.grpo_logprob_loss_fwd_bwd``: ``kl_kind``, ``kl_coef``, ``ref_logp`` (input order, all
    tokens), ``ent_coef`` and ``entropy_tok`` (input order, all tokens; written).

    ``logits_host`` (instead of ``logits``): the batch's logits in host memory, exec order. Each
    optimizer step's rows are streamed in one ``grpo_logprob_loss_fwd_bwd_host`` call through
    ``staging`` (device, 2 * block_rows rows), the copies on ``copy_stream``. The micro-batch
    boundaries change no bit, so the step is one call; ``chunk_ready`` and ``side_stream`` do
    not apply, and ``launch_events`` receives one pair per step.

    ``side_stream`` (optional, a stream or a list of streams): the chunks of a step rotate
    between ``stream`` and these streams, so that the next chunk's blocks take the SMs the
    current chunk's last rows leave idle. Chunks of a step write disjoint rows and only add to
    the step's integer counters, so the results are the same bits; the step's finish waits for
    every stream.

    ``finish_stream`` (optional, with device logits): each optimizer step's finish runs on this
    stream, after that step's chunks on every stream, while the next step's chunks go on; the
    caller's stream waits for the last finish at the end. A finish reads only its own step's
    per-token losses and accumulator (and, deferred, scales its own step's dlogits rows), so
    the results are the same bits."""
    import torch

    # checks that need no device, made before anything is enqueued
    p = bp.plan
    need = int(p["n_steps"]) * _lib.ACC_BYTES
    if accs.numel() * accs.element_size() < need:
        raise ValueError(f"accs must hold {need} bytes (one accumulator per optimizer step)")
    if agg == _lib.AGG_SEQ_MEAN_TOKEN_MEAN and w_tok is None:
        raise ValueError("SEQ_MEAN_TOKEN_MEAN needs the per-token weights w_tok")
    st = torch.cuda.current_stream() if stream is None else stream
    sides = [] if side_stream is None else (list(side_stream) if isinstance(side_stream, (list, tuple))
                                            else [side_stream])
    fs = finish_stream if logits_host is None else None
    rotation = [st] + sides
    launches = 0
    if rewards is not None:
        _lib.grpo_group_advantage(rewards, group_size, adv_eps, True, adv_rollout, row_rollout,
                                  row_tok_off, adv_tok, stream=st)
        launches += 2
    plain = agg == _lib.AGG_TOKEN_MEAN and w_tok is None
    # each step's divisor D and its grad scale 1/max(D, 1), both from the library
    divisors, _, scales = _lib.grpo_plan_token_weights(p, bp.row_len, bp.row_valid, agg, want_w=False,
                                                       want_scale=True)
    for s in range(p["n_steps"]):
        N = int(p["step_valid_tokens"][s])
        D = int(divisors[s])
        scale = 1.0 if deferred else float(scales[s])
        acc = accs[s * _lib.ACC_BYTES:(s + 1) * _lib.ACC_BYTES]
        if logits_host is not None:
            launches += _host_step(bp, s, logits_host, staging, block_rows, copy_stream, st, dlogits, target,
                                   old_logp, adv_tok, mask, loss_tok, logp_tok, acc, clip_eps, scale, tok_src,
                                   w_tok, terms, V, launch_events)
        elif s == 0 or fs is None:
            for ss in sides:
                ss.wait_stream(st)  # the advantage (and, without a finish stream, the previous finish)
        chunks = range(0) if logits_host is not None else range(p["step_chunk_off"][s], p["step_chunk_off"][s + 1])
        for i, c in enumerate(chunks):
            a, b = int(bp.exec_tok_off[c]), int(bp.exec_tok_off[c + 1])
            cs = rotation[i % len(rotation)]
            if chunk_ready is not None:
                cs.wait_event(chunk_ready[c])
            if b == a:
                continue
            if launch_events is not None:
                e0 = torch.cuda.Event(enable_timing=True)
                e0.record(cs)
            if tok_src is None:
                # exec order == input order: the chunk's side inputs are the same slice
                side = (target[a:b], None if old_logp is None else old_logp[a:b], adv_tok[a:b],
                        mask[a:b], loss_tok[a:b], None if logp_tok is None else logp_tok[a:b], None,
                        None if w_tok is None else w_tok[a:b])
            else:
                # side arrays stay whole; the kernel reads them through the token index
                side = (target, old_logp, adv_tok, mask, loss_tok, logp_tok, tok_src[a:b], w_tok)
            tg, od, ad, mk, lt, lp, ts, wt = side
            ct = None
            if terms is not None or wt is not None:
                ct = dict(terms or {})
                if tok_src is None:  # the per-token arrays of the terms follow the chunk's slice
                    for k in ("ref_logp", "entropy_tok"):
                        if ct.get(k) is not None:
                            ct[k] = ct[k][a:b]
                if wt is not None:
                    ct["w_tok"] = wt
            _lib.grpo_logprob_loss_fwd_bwd(
                logits[a:b], tg, od, ad, mk, clip_eps, scale,
                None if dlogits is None else dlogits[a:b], lt, lp, acc, tok_src=ts, V=V, stream=cs,
                terms=ct)
            if launch_events is not None:
                e1 = torch.cuda.Event(enable_timing=True)
                e1.record(cs)
                launch_events.append((e0, e1))
            launches += 1
        fin = st
        if fs is not None:
            fs.wait_stream(st)  # this step's chunks on every stream
            for ss in sides:
                fs.wait_stream(ss)
            fin = fs
        elif logits_host is None:
            for ss in sides:
                st.wait_stream(ss)
        t0, t1 = bp.step_tok_range[s]
        e0, e1 = bp.step_exec_range[s]
        grads = [] if dlogits is None or e1 == e0 else [dlogits[e0:e1]]
        if plain:
            _lib.grpo_finish_step(acc, loss_tok[t0:t1], expected_N=N, deferred=deferred,
                                  grad_bufs=grads, sync=False, stream=fin)
        else:
            _lib.grpo_finish_step_ex(acc, loss_tok[t0:t1], None if w_tok is None else w_tok[t0:t1],
                                     divisor=D, expected_N=N, deferred=deferred, grad_bufs=grads,
                                     sync=False, stream=fin)
        launches += 1 + len(grads)
    if fs is not None:
        st.wait_stream(fs)
        for ss in sides:
            st.wait_stream(ss)
    return launches


def _host_step(bp, s, logits_host, staging, block_rows, copy_stream, st, dlogits, target, old_logp, adv_tok,
               mask, loss_tok, logp_tok, acc, clip_eps, scale, tok_src, w_tok, terms, V, launch_events) -> int:
    """One optimizer step's rows streamed from host memory: returns the kernel launches."""
    import torch

    e0, e1 = bp.step_exec_range[s]
    if e1 == e0:
        return 0
    ct = dict(terms or {})
    if w_tok is not None:
        ct["w_tok"] = w_tok
    if tok_src is None:  # exec order == input order: the side arrays follow the rows
        side = [None if a is None else a[e0:e1] for a in (target, old_logp, adv_tok, mask, loss_tok, logp_tok)]
        for k in ("ref_logp", "entropy_tok", "w_tok"):
            if ct.get(k) is not None:
                ct[k] = ct[k][e0:e1]
        ts = None
    else:
        side = [target, old_logp, adv_tok, mask, loss_tok, logp_tok]
        ts = tok_src[e0:e1]
    tg, od, ad, mk, lt, lp = side
    if launch_events is not None:
        ev0 = torch.cuda.Event(enable_timing=True)
        ev0.record(st)
    _lib.grpo_logprob_loss_fwd_bwd_host(logits_host[e0:e1], tg, od, ad, mk, clip_eps, scale,
                                        None if dlogits is None else dlogits[e0:e1], lt, lp, acc, staging,
                                        block_rows, tok_src=ts, V=V, stream=st, copy_stream=copy_stream,
                                        terms=ct or None)
    if launch_events is not None:
        ev1 = torch.cuda.Event(enable_timing=True)
        ev1.record(st)
        launch_events.append((ev0, ev1))
    return -(-(e1 - e0) // block_rows)


def read_results(accs, n_steps: int) -> List[dict]:
    raw = accs.view(n_steps, _lib.ACC_BYTES)[:, 64:].cpu().numpy()
    return [_lib.grpo_step_result.from_buffer_copy(raw[s].tobytes()).as_dict() for s in range(n_steps)]


# ---- data parallelism over one optimizer step's rows ------------------------------------------
#
# Every rank plans the whole batch (the planner is host-only and cheap), so each rank knows
# every step's N without communication. Rank r runs the rows `dp_row_block` gives it, with
# grad_scale = 1/max(N, 1) and a finish whose divisor is N (grpo_finish_step_ex); its dlogits
# rows are then those of a single-GPU run. The step's one exchange is the ranks' float64 loss
# sums and integer counts (`dp_allreduce_step_result`).

_RESULT_FIELDS = ("loss_sum", "n_valid", "n_clipped", "n_nonfinite", "n_tokens", "status", "kernel_flags")


def dp_row_block(n_rows: int, rank: int, world: int) -> tuple:
    """The contiguous rows [lo, hi) of an optimizer step's `n_rows` that data-parallel rank
    `rank` of `world` runs: equal counts, the first n_rows % world ranks one row more."""
    if world < 1 or not 0 <= rank < world or n_rows < 0:
        raise ValueError("need 0 <= rank < world and n_rows >= 0")
    q, r = divmod(n_rows, world)
    lo = rank * q + min(rank, r)
    return lo, lo + q + (1 if rank < r else 0)


def dp_exec_ranges(bp: BatchPlan, s: int, rank: int, world: int) -> List[tuple]:
    """The exec-order token ranges [t0, t1) of optimizer step `s` that data-parallel rank
    `rank` of `world` runs.

    A compaction plan assigns rows to GPUs itself: each padded group is split evenly across
    the GPUs ("How a context-compaction step fits a variable number of rows into one batch",
    the figure), in the plan's ``row_gpu``. The plan must then have been made for `world`
    GPUs. Any other plan splits the step's rows, in execution order, into `dp_row_block`'s
    contiguous blocks."""
    p = bp.plan
    c0, c1 = int(p["step_chunk_off"][s]), int(p["step_chunk_off"][s + 1])
    j0, j1 = int(p["chunk_row_off"][c0]), int(p["chunk_row_off"][c1])
    lens = bp.row_len[np.asarray(p["row_src"][j0:j1], np.int64)]
    off = int(bp.exec_tok_off[c0]) + np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    if int(p["q"]) > 0:
        gpu = np.asarray(p["row_gpu"][j0:j1])
        n_gpus = int(np.asarray(p["row_gpu"][:int(p["n_rows"])]).max()) + 1
        if n_gpus != world:
            raise ValueError(f"the compaction plan was made for {n_gpus} GPUs, not {world}")
        ranges, j = [], 0
        while j < j1 - j0:
            if gpu[j] != rank:
                j += 1
                continue
            k = j
            while k < j1 - j0 and gpu[k] == rank:
                k += 1
            ranges.append((int(off[j]), int(off[k])))
            j = k
        return ranges
    lo, hi = dp_row_block(j1 - j0, rank, world)
    return [(int(off[lo]), int(off[hi]))] if hi > lo else []


def combine_step_results(results: List[dict], divisor: int) -> dict:
    """One step's result from the per-rank results of its row blocks (each finished with the
    step's divisor), by grpo_combine_step_results: float64 loss sums and counts added in rank
    order, loss = sum / max(divisor, 1), the first error status, OR-ed kernel flags."""
    return _lib.grpo_combine_step_results(results, divisor)


def dp_allreduce_step_result(res: dict, divisor: int, group=None) -> dict:
    """Every rank's step result -> the whole step's, identical on all ranks: one all-gather of
    seven numbers per rank (float64; the counts are exact below 2^53), then
    `combine_step_results` in rank order. CPU tensors under gloo, device tensors under nccl."""
    import torch
    import torch.distributed as dist

    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend(group) == "nccl" else "cpu"
    mine = torch.tensor([float(res[k]) for k in _RESULT_FIELDS], dtype=torch.float64, device=dev)
    allv = [torch.empty_like(mine) for _ in range(dist.get_world_size(group))]
    dist.all_gather(allv, mine, group=group)
    rows = [dict(zip(_RESULT_FIELDS, v.cpu().tolist())) for v in allv]
    return combine_step_results(rows, divisor)
