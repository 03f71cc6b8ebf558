"""Oracle batch planner (integer only): one collected batch -> optimizer steps -> chunks.

Test infrastructure only; see ``oracle/__init__.py``.

Sources, cited by page title and section:

* "Sizing mini-batches and micro-batches" (cosmos posttrain batching how-to):
  - *The config surface*: ``batch`` must be a positive multiple of ``group_size``;
    ``mini = 0`` means the whole batch, ``micro = 0`` means one chunk; ``n_mini = batch/mini``,
    ``n_micro = mini/micro``; exact divisibility is required at every level.
  - *A worked example*: 32 trajectories, mini 16, micro 8 -> a 2x2 loop of four calls.
  - *The hard part: deferred normalization*: N counts masked completion positions; one
    divisor per optimizer step.
  - *pi_old must be frozen across the window*: the ahead pass is needed when
    ``n_mini > 1`` and the rollout log-probs are not used for the loss.
* "22-mini-batch-micro-batch-dynamic-batch-size的区别" (verl batching article), section 3
  (dynamic batch size): every row must fit ``max_token_len``; the bin count is the total
  tokens over the budget, rounded up; rows are binned by an estimated workload; small bins may
  go to both ends; an index map restores the original order.
* "How a context-compaction step fits a variable number of rows into one batch" (NeMo-RL
  explainer), the figure and *What it costs*: each group is padded up to a multiple of
  ``Q = n_gpus * lcm(micro, logprob_batch)`` with masked, reward-0 copies of a real row; each
  group is split evenly across the GPUs; the step must hold exactly ``batch`` rollouts;
  compaction rejects sequence packing, dynamic batching and the interleaved pipeline;
  one optimizer step per training step.

Readings where the pages are silent:

* fixed chunks are contiguous and unshuffled, in input order;
* a pad row copies the input of its group's FIRST real row;
* GPU slot of the k-th row of a padded group of P rows is ``k // (P // n_gpus)``
  (contiguous blocks, which is also what the explainer's figure draws);
* compaction runs one optimizer step, so ``mini`` must be 0 or ``batch``;
* the dynamic binning rule (longest-processing-time greedy with a capacity check) is ours:
  the pages name no partition algorithm. Where the budget does not bind, the rule is plain
  LPT list scheduling, and the tests pin it there to Graham's tight instance (heaviest bin
  4k-1 against the optimum 3k) and to his 4/3 - 1/(3k) bound against brute force.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

# Status codes of the planner (same numbers as the library's public header; restated here
# so that the oracle depends on nothing outside this package).
OK = 0
ERR_INVALID = -1
ERR_DIVISIBILITY = -2
ERR_ROLLOUT_COUNT = -3
ERR_TOKEN_BUDGET = -4
ERR_INCOMPATIBLE = -5

WORKLOAD_TOKENS = 0     # w = L
WORKLOAD_ATTENTION = 1  # w = L * L


class PlanError(Exception):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} (code {code})")
        self.code = code


@dataclass
class PlanConfig:
    batch: int = 32            # rollouts per replica per loop step
    mini: int = 0              # rollouts per optimizer step; 0 = whole batch
    micro: int = 0             # rollouts (rows, under compaction) per chunk; 0 = one chunk
    group_size: int = 1
    dynamic: int = 0           # token-budget binning inside each mini-batch
    max_token_len: int = 0
    workload: int = WORKLOAD_TOKENS
    min_bins: int = 0
    bin_multiple: int = 1
    balance_ends: int = 0
    compaction: int = 0        # context compaction: rollouts may span several rows
    n_gpus: int = 1
    logprob_batch: int = 1
    sequence_packing: int = 0
    interleaved_pipeline: int = 0
    use_rollout_logprobs: int = 0


@dataclass
class Plan:
    n_rows: int = 0
    n_chunks: int = 0
    n_steps: int = 0
    n_micro: int = 0           # chunks per step when constant, else 0
    q: int = 0                 # compaction multiple Q, else 0
    n_pad_rows: int = 0
    needs_old_logp_cache: int = 0
    row_src: List[int] = field(default_factory=list)      # input row feeding exec row j
    row_pad: List[int] = field(default_factory=list)      # 1 for padding rows
    row_gpu: List[int] = field(default_factory=list)      # GPU slot (compaction), else 0
    row_rollout: List[int] = field(default_factory=list)  # rollout of exec row, -1 for pad
    inv_perm: List[int] = field(default_factory=list)     # exec position of input row i
    chunk_row_off: List[int] = field(default_factory=list)
    step_chunk_off: List[int] = field(default_factory=list)
    step_in_row_off: List[int] = field(default_factory=list)  # input rows of each step
    chunk_tokens: List[int] = field(default_factory=list)
    step_valid_tokens: List[int] = field(default_factory=list)  # N of each step
    step_valid_rows: List[int] = field(default_factory=list)


def _ceil_div(a: int, b: int) -> int:
    return -((-a) // b)


def _round_up(a: int, m: int) -> int:
    return _ceil_div(a, m) * m if m > 1 else a


def plan(cfg: PlanConfig, row_len, row_valid, seg_counts=None, n_rollouts: Optional[int] = None) -> Plan:
    """Plan one collected batch.

    ``row_len[i]``   -- token rows (logits rows) of input row i.
    ``row_valid[i]`` -- mask=1 positions of input row i (policy_len), 0 <= valid <= len.
    ``seg_counts[r]``-- rows produced by rollout r (compaction only).
    ``n_rollouts``   -- rollouts actually collected (defaults to len(seg_counts) or rows).
    Raises PlanError with one of the status codes above.
    """
    row_len = [int(x) for x in row_len]
    row_valid = [int(x) for x in row_valid]
    n_in = len(row_len)
    if len(row_valid) != n_in:
        raise PlanError(ERR_INVALID, "row_len and row_valid differ in length")
    for L, v in zip(row_len, row_valid):
        if L < 0 or v < 0 or v > L:
            raise PlanError(ERR_INVALID, "row lengths must satisfy 0 <= valid <= len")
    if cfg.batch <= 0 or cfg.group_size <= 0 or cfg.mini < 0 or cfg.micro < 0:
        raise PlanError(ERR_INVALID, "batch and group_size must be positive, mini/micro >= 0")
    # The config surface: batch is a positive multiple of group_size.
    if cfg.batch % cfg.group_size != 0:
        raise PlanError(ERR_DIVISIBILITY, "batch must be a multiple of group_size")

    if cfg.compaction:
        return _plan_compaction(cfg, row_len, row_valid, seg_counts, n_rollouts)

    if n_rollouts is None:
        n_rollouts = n_in
    # One row per rollout outside compaction; the step needs exactly `batch` of them.
    if n_rollouts != cfg.batch or n_in != cfg.batch:
        raise PlanError(ERR_ROLLOUT_COUNT, "the batch must hold exactly `batch` rollouts")

    mini = cfg.mini if cfg.mini else cfg.batch
    micro = cfg.micro if cfg.micro else mini
    if cfg.batch % mini != 0 or mini % micro != 0:
        raise PlanError(ERR_DIVISIBILITY, "batch % mini and mini % micro must be 0")
    n_mini = cfg.batch // mini

    p = Plan()
    p.n_steps = n_mini
    p.row_src = list(range(n_in))
    p.row_pad = [0] * n_in
    p.row_gpu = [0] * n_in
    p.row_rollout = list(range(n_in))
    p.n_rows = n_in
    p.step_in_row_off = [i * mini for i in range(n_mini + 1)]

    if not cfg.dynamic:
        n_micro = mini // micro
        p.n_micro = n_micro
        p.chunk_row_off = [c * micro for c in range(n_mini * n_micro + 1)]
        p.step_chunk_off = [i * n_micro for i in range(n_mini + 1)]
    else:
        if cfg.max_token_len <= 0:
            raise PlanError(ERR_INVALID, "dynamic batching needs max_token_len > 0")
        if max(row_len) > cfg.max_token_len:
            raise PlanError(ERR_TOKEN_BUDGET, "a row is longer than max_token_len")
        order: List[int] = []
        p.chunk_row_off = [0]
        p.step_chunk_off = [0]
        for i in range(n_mini):
            rows = list(range(i * mini, (i + 1) * mini))
            bins = _dynamic_bins(cfg, rows, row_len)
            for b in bins:
                order.extend(b)
                p.chunk_row_off.append(len(order))
            p.step_chunk_off.append(len(p.chunk_row_off) - 1)
        p.row_src = order
        p.row_rollout = list(order)
        p.n_micro = 0

    return _finish(cfg, p, row_len, row_valid, n_in)


def _dynamic_bins(cfg: PlanConfig, rows: List[int], row_len: List[int]) -> List[List[int]]:
    """Token-budget bins of one mini-batch (verl batching article, section 3).

    1. k = max(ceil(sum L / max_token_len), min_bins, 1), rounded up to bin_multiple, capped
       at the number of rows.
    2. workload w = L (tokens) or L*L (attention pressure).
    3. visit rows by (w desc, L desc, index asc); put each into the feasible bin (tokens + L
       <= max_token_len) with the least (workload, tokens, bin index); if none is feasible,
       grow k (next multiple of bin_multiple, capped at the row count) and start over.
    4. rows inside a bin by index; bins by their smallest row (empty bins last);
       optionally the small bins at both ends: sort by (workload, smallest row) ascending and
       place them at positions 0, k-1, 1, k-2, ...
    """
    B = len(rows)
    cap = cfg.max_token_len
    total = sum(row_len[r] for r in rows)
    k = max(_ceil_div(total, cap), cfg.min_bins, 1)
    k = _round_up(k, cfg.bin_multiple)
    k = min(k, B)

    def weight(r):
        L = row_len[r]
        return L * L if cfg.workload == WORKLOAD_ATTENTION else L

    visit = sorted(rows, key=lambda r: (-weight(r), -row_len[r], r))
    while True:
        load_w = [0] * k
        load_t = [0] * k
        members: List[List[int]] = [[] for _ in range(k)]
        ok = True
        for r in visit:
            best = -1
            for b in range(k):
                if load_t[b] + row_len[r] > cap:
                    continue
                if best < 0 or (load_w[b], load_t[b], b) < (load_w[best], load_t[best], best):
                    best = b
            if best < 0:
                ok = False
                break
            members[best].append(r)
            load_w[best] += weight(r)
            load_t[best] += row_len[r]
        if ok:
            break
        assert k < B, "k = number of rows is always feasible"
        k = min(_round_up(k + 1, cfg.bin_multiple), B)

    for m in members:
        m.sort()
    big = float("inf")
    bins = list(range(k))
    bins.sort(key=lambda b: (members[b][0] if members[b] else big, b))
    if cfg.balance_ends:
        asc = sorted(bins, key=lambda b: (load_w[b], members[b][0] if members[b] else big, b))
        placed = [None] * k
        lo, hi = 0, k - 1
        for idx, b in enumerate(asc):
            if idx % 2 == 0:
                placed[lo] = b
                lo += 1
            else:
                placed[hi] = b
                hi -= 1
        bins = placed
    return [members[b] for b in bins]


def _plan_compaction(cfg, row_len, row_valid, seg_counts, n_rollouts) -> Plan:
    """Context compaction (NeMo-RL explainer): pad every group to a multiple of Q."""
    if cfg.dynamic or cfg.sequence_packing or cfg.interleaved_pipeline:
        raise PlanError(ERR_INCOMPATIBLE,
                        "compaction rejects dynamic batching, sequence packing, interleaved pipeline")
    if cfg.mini not in (0, cfg.batch):
        raise PlanError(ERR_INCOMPATIBLE, "compaction takes one optimizer step per training step")
    if seg_counts is None:
        raise PlanError(ERR_INVALID, "compaction needs seg_counts")
    seg_counts = [int(s) for s in seg_counts]
    if cfg.micro <= 0 or cfg.n_gpus <= 0 or cfg.logprob_batch <= 0:
        raise PlanError(ERR_INVALID, "compaction needs micro, n_gpus, logprob_batch >= 1")
    if any(s < 1 for s in seg_counts) or sum(seg_counts) != len(row_len):
        raise PlanError(ERR_INVALID, "seg_counts must be >= 1 and sum to the row count")
    if n_rollouts is None:
        n_rollouts = len(seg_counts)
    if n_rollouts != len(seg_counts) or n_rollouts != cfg.batch:
        raise PlanError(ERR_ROLLOUT_COUNT, "the step must hold exactly `batch` rollouts")

    lcm = cfg.micro * cfg.logprob_batch // math.gcd(cfg.micro, cfg.logprob_batch)
    Q = cfg.n_gpus * lcm
    G = cfg.group_size
    n_groups = cfg.batch // G

    first_row_of_rollout = [0] * (cfg.batch + 1)
    for r in range(cfg.batch):
        first_row_of_rollout[r + 1] = first_row_of_rollout[r] + seg_counts[r]

    p = Plan()
    p.q = Q
    for g in range(n_groups):
        real = []  # (input row, rollout) in rollout-then-segment order
        for r in range(g * G, (g + 1) * G):
            for s in range(seg_counts[r]):
                real.append((first_row_of_rollout[r] + s, r))
        padded = _ceil_div(len(real), Q) * Q
        per_gpu = padded // cfg.n_gpus
        src0 = real[0][0]
        for k in range(padded):
            if k < len(real):
                p.row_src.append(real[k][0])
                p.row_rollout.append(real[k][1])
                p.row_pad.append(0)
            else:
                p.row_src.append(src0)   # copies the group's first real row's input
                p.row_rollout.append(-1)
                p.row_pad.append(1)
            p.row_gpu.append(k // per_gpu)
    p.n_rows = len(p.row_src)
    p.n_pad_rows = sum(p.row_pad)
    n_chunks = p.n_rows // cfg.micro
    p.chunk_row_off = [c * cfg.micro for c in range(n_chunks + 1)]
    p.step_chunk_off = [0, n_chunks]
    p.n_steps = 1
    p.n_micro = n_chunks
    p.step_in_row_off = [0, len(row_len)]
    return _finish(cfg, p, row_len, row_valid, len(row_len))


def _finish(cfg, p: Plan, row_len, row_valid, n_in) -> Plan:
    p.n_chunks = len(p.chunk_row_off) - 1
    p.inv_perm = [-1] * n_in
    for j, (src, pad) in enumerate(zip(p.row_src, p.row_pad)):
        if not pad:
            p.inv_perm[src] = j
    p.chunk_tokens = []
    for c in range(p.n_chunks):
        a, b = p.chunk_row_off[c], p.chunk_row_off[c + 1]
        p.chunk_tokens.append(sum(row_len[p.row_src[j]] for j in range(a, b)))
    p.step_valid_tokens = []
    p.step_valid_rows = []
    for i in range(p.n_steps):
        a = p.chunk_row_off[p.step_chunk_off[i]]
        b = p.chunk_row_off[p.step_chunk_off[i + 1]]
        n_tok = 0
        n_row = 0
        for j in range(a, b):
            if p.row_pad[j]:
                continue  # padding rows are masked: they add no valid token and no row
            v = row_valid[p.row_src[j]]
            n_tok += v
            n_row += 1 if v > 0 else 0
        p.step_valid_tokens.append(n_tok)
        p.step_valid_rows.append(n_row)
    p.needs_old_logp_cache = 1 if (p.n_steps > 1 and not cfg.use_rollout_logprobs) else 0
    return p


def restore(plan_: Plan, exec_values):
    """Undo the execution order: value of input row i = exec_values[inv_perm[i]]."""
    return [exec_values[j] for j in plan_.inv_perm]
