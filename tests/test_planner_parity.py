"""Host planner in the C-ABI library vs the oracle planner: bit-exact on every field and on
every error code. Host code only: no GPU needed."""
import numpy as np
import pytest

from oracle import planner as OP
from rl_post_token_gb300 import workloads as W

FIELDS = ["row_src", "row_pad", "row_gpu", "row_rollout", "inv_perm", "chunk_row_off",
          "step_chunk_off", "step_in_row_off", "chunk_tokens", "step_valid_tokens", "step_valid_rows"]
SCALARS = ["n_rows", "n_chunks", "n_steps", "n_micro", "q", "n_pad_rows", "needs_old_logp_cache"]


def _both(cfg, row_len, row_valid, seg=None, n_rollouts=None):
    from rl_post_token_gb300 import _lib
    try:
        o = OP.plan(OP.PlanConfig(**cfg), row_len, row_valid, seg_counts=seg, n_rollouts=n_rollouts)
        o_code = 0
    except OP.PlanError as e:
        o, o_code = None, e.code
    try:
        c = _lib.grpo_plan_microbatches(cfg, row_len, row_valid, seg_counts=seg, n_rollouts=n_rollouts)
        c_code = 0
    except _lib.GrpoError as e:
        c, c_code = None, e.code
    return o, o_code, c, c_code


def _assert_same(cfg, row_len, row_valid, seg=None, n_rollouts=None):
    o, oc, c, cc = _both(cfg, row_len, row_valid, seg, n_rollouts)
    assert oc == cc, (cfg, oc, cc)
    if oc:
        return None
    for k in SCALARS:
        assert getattr(o, k) == c[k], k
    for k in FIELDS:
        assert np.array_equal(np.asarray(getattr(o, k), np.int64), c[k].astype(np.int64)), k
    return c


@pytest.mark.parametrize("name", ["tiny", "qwen_step", "dynamic", "compaction"])
def test_workload_plans(grpo_lib, name):
    wl = W.make_workload(name)
    c = _assert_same(wl.plan, wl.row_len, wl.row_valid, wl.seg_counts)
    assert c is not None
    assert int(c["step_valid_tokens"].sum()) == wl.n_valid


def test_compaction_example_numbers(grpo_lib):
    wl = W.make_workload("compaction")
    c = _assert_same(wl.plan, wl.row_len, wl.row_valid, wl.seg_counts)
    assert (c["n_rows"], c["n_pad_rows"], c["q"], c["n_chunks"]) == (16, 3, 4, 16)


@pytest.mark.parametrize("seed", range(40))
def test_random_fixed_and_dynamic(grpo_lib, seed):
    rng = np.random.default_rng(seed)
    G = int(rng.choice([1, 2, 4, 8]))
    B = G * int(rng.integers(1, 17))
    row_len = rng.integers(0, 3000, B)
    row_valid = (row_len * rng.random(B)).astype(np.int64)
    cfg = dict(batch=B, group_size=G, mini=int(rng.choice([0, B, B // 2 if B % 2 == 0 else B])),
               micro=int(rng.choice([0, 1, 2, 4])), use_rollout_logprobs=int(rng.integers(0, 2)))
    if rng.random() < 0.5:
        cfg.update(dynamic=1, max_token_len=int(rng.choice([2999, 4096, 8192, 20000])),
                   workload=int(rng.integers(0, 2)), min_bins=int(rng.integers(0, 5)),
                   bin_multiple=int(rng.choice([1, 2, 3])), balance_ends=int(rng.integers(0, 2)))
    _assert_same(cfg, row_len, row_valid)


@pytest.mark.parametrize("seed", range(30))
def test_random_compaction(grpo_lib, seed):
    rng = np.random.default_rng(500 + seed)
    G = int(rng.choice([1, 2, 4]))
    n_groups = int(rng.integers(1, 6))
    B = G * n_groups
    seg = rng.integers(1, 6, B)
    rows = int(seg.sum())
    row_len = rng.integers(1, 2048, rows)
    cfg = dict(batch=B, group_size=G, compaction=1, micro=int(rng.choice([1, 2, 3])),
               n_gpus=int(rng.choice([1, 2, 4, 8])), logprob_batch=int(rng.choice([1, 2, 4])))
    _assert_same(cfg, row_len, row_len, seg)


@pytest.mark.parametrize("case", [
    (dict(batch=30, group_size=4), 30, None),
    (dict(batch=32, group_size=4, mini=12), 32, None),
    (dict(batch=32, group_size=4, mini=16, micro=6), 32, None),
    (dict(batch=32, group_size=4), 28, None),
    (dict(batch=0, group_size=4), 4, None),
    (dict(batch=8, group_size=4, dynamic=1, max_token_len=100), 8, None),
    (dict(batch=8, group_size=4, dynamic=1, max_token_len=0), 8, None),
    (dict(batch=6, group_size=2, compaction=1, micro=1, n_gpus=4, dynamic=1, max_token_len=9999), 13, [1, 3, 2, 5, 1, 1]),
    (dict(batch=6, group_size=2, compaction=1, micro=1, n_gpus=4, sequence_packing=1), 13, [1, 3, 2, 5, 1, 1]),
    (dict(batch=6, group_size=2, compaction=1, micro=1, n_gpus=4, mini=2), 13, [1, 3, 2, 5, 1, 1]),
    (dict(batch=6, group_size=2, compaction=1, micro=1, n_gpus=4), 12, [1, 3, 2, 5, 1]),
    (dict(batch=6, group_size=2, compaction=1, micro=0, n_gpus=4), 13, [1, 3, 2, 5, 1, 1]),
    (dict(batch=6, group_size=2, compaction=1, micro=1, n_gpus=4), 12, [1, 3, 2, 5, 1, 0]),
])
def test_error_codes_agree(grpo_lib, case):
    cfg, rows, seg = case
    row_len = [120] * rows
    _, oc, _, cc = _both(cfg, row_len, row_len, seg)
    assert oc == cc and oc < 0


def test_token_index(grpo_lib):
    from rl_post_token_gb300 import _lib
    wl = W.make_workload("compaction", row_tokens=3)
    p = _lib.grpo_plan_microbatches(wl.plan, wl.row_len, wl.row_valid, wl.seg_counts)
    idx = _lib.grpo_plan_token_index(p, wl.row_len)
    assert idx.shape[0] == 16 * 3
    off = wl.tok_off
    want = []
    for j in range(p["n_rows"]):
        r = p["row_src"][j]
        toks = list(range(off[r], off[r + 1]))
        want += [-1 - t for t in toks] if p["row_pad"][j] else toks
    assert idx.tolist() == want


@pytest.mark.parametrize("k", [2, 3, 4, 6])
@pytest.mark.parametrize("workload", [0, 1])
def test_dynamic_graham_instances(grpo_lib, k, workload):
    # Graham's tight LPT instance (two rows each of 2k-1 .. k+1 tokens, three of k) with the
    # token budget out of the way and k bins forced; both workload estimates
    row_len = [L for L in range(2 * k - 1, k, -1) for _ in range(2)] + [k] * 3
    n = len(row_len)
    cfg = dict(batch=n, group_size=1, dynamic=1, max_token_len=sum(row_len), min_bins=k, workload=workload)
    c = _assert_same(cfg, row_len, row_len)
    assert c["n_chunks"] == k
    if workload == 0:
        assert int(c["chunk_tokens"].max()) == 4 * k - 1
