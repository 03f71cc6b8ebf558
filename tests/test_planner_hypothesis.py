"""Randomised search (hypothesis) for any input on which the library's host code and the
oracle disagree: the planner (every field and every error code, over fixed, dynamic and
compaction configurations), the token index, the aggregation weights and the accumulation
window. Host code only."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
from hypothesis import HealthCheck, given, settings  # noqa: E402

from tests.test_planner_parity import _assert_same  # noqa: E402


@st.composite
def fixed_or_dynamic(draw):
    G = draw(st.sampled_from([1, 2, 3, 4, 8]))
    B = G * draw(st.integers(1, 12))
    row_len = draw(st.lists(st.integers(0, 5000), min_size=B, max_size=B))
    row_valid = [draw(st.integers(0, L)) for L in row_len]
    cfg = dict(batch=B, group_size=G, mini=draw(st.sampled_from([0, B, B // 2, 3, G])),
               micro=draw(st.sampled_from([0, 1, 2, 3, 4])),
               use_rollout_logprobs=draw(st.integers(0, 1)))
    if draw(st.booleans()):
        cfg.update(dynamic=1, max_token_len=draw(st.integers(1, 12000)),
                   workload=draw(st.integers(0, 1)), min_bins=draw(st.integers(0, 6)),
                   bin_multiple=draw(st.integers(0, 4)), balance_ends=draw(st.integers(0, 1)))
    return cfg, row_len, row_valid


@st.composite
def compaction(draw):
    G = draw(st.sampled_from([1, 2, 4]))
    n_groups = draw(st.integers(1, 5))
    B = G * n_groups
    seg = draw(st.lists(st.integers(0, 6), min_size=B, max_size=B))
    rows = int(sum(seg))
    row_len = draw(st.lists(st.integers(1, 3000), min_size=rows, max_size=rows))
    cfg = dict(batch=draw(st.sampled_from([B, B + G])), group_size=G, compaction=1,
               micro=draw(st.integers(0, 4)), n_gpus=draw(st.integers(0, 8)),
               logprob_batch=draw(st.integers(0, 4)), mini=draw(st.sampled_from([0, B, 1])))
    return cfg, row_len, seg


SETTINGS = dict(max_examples=400, deadline=None, suppress_health_check=[HealthCheck.too_slow])


@settings(**SETTINGS)
@given(fixed_or_dynamic())
def test_fixed_and_dynamic_plans_agree(grpo_lib, case):
    cfg, row_len, row_valid = case
    _assert_same(cfg, np.asarray(row_len), np.asarray(row_valid))


@settings(**SETTINGS)
@given(compaction())
def test_compaction_plans_agree(grpo_lib, case):
    cfg, row_len, seg = case
    _assert_same(cfg, np.asarray(row_len), np.asarray(row_len), seg)


@st.composite
def window_runs(draw):
    n_micro = draw(st.integers(1, 8))
    chunks = draw(st.lists(st.tuples(st.booleans(), st.floats(-1e6, 1e6, allow_nan=False, width=64),
                                     st.integers(0, 5000)), min_size=0, max_size=60))
    return n_micro, chunks


@settings(**SETTINGS)
@given(window_runs())
def test_window_runs_agree(grpo_lib, run):
    # the host accumulation window: every chunk's action and scale, the counters and the
    # roll-up, for any sequence of finite and non-finite chunks
    import math

    from oracle import window as OW
    from rl_post_token_gb300 import _lib
    n_micro, chunks = run
    o, c = OW.Window(n_micro), _lib.Window(n_micro)
    for finite, loss, denom in chunks:
        x = loss if finite else math.nan
        assert o.chunk(finite, x, denom) == c.grpo_window_chunk(finite, x, denom)
    st_ = c.state
    assert (st_["steps"], st_["skipped_windows"], st_["dropped_chunks"]) == (o.steps, o.skipped_windows,
                                                                             o.dropped_chunks)
    lo, do, so = o.rollup()
    lc, dc, sc = c.grpo_window_rollup()
    assert (do, so) == (dc, sc)
    assert lc == lo or abs(lc - lo) <= 1e-15 * max(abs(lo), 1e-300)


@st.composite
def weight_plans(draw):
    G = draw(st.sampled_from([1, 2, 4]))
    B = G * draw(st.integers(1, 10))
    row_len = draw(st.lists(st.integers(0, 60), min_size=B, max_size=B))
    row_valid = [draw(st.integers(0, L)) for L in row_len]
    mini = draw(st.sampled_from([d for d in range(1, B + 1) if B % d == 0]))
    cfg = dict(batch=B, group_size=G, mini=mini, micro=draw(st.sampled_from([d for d in range(1, mini + 1)
                                                                              if mini % d == 0])))
    if draw(st.booleans()):
        cfg.update(dynamic=1, max_token_len=max(row_len + [1]) + draw(st.integers(0, 200)),
                   workload=draw(st.integers(0, 1)), balance_ends=draw(st.integers(0, 1)))
    return cfg, row_len, row_valid


@settings(**SETTINGS)
@given(weight_plans(), st.sampled_from([0, 1, 2]))
def test_aggregation_weights_agree(grpo_lib, case, agg):
    # grpo_plan_token_weights: every step's divisor and every token's weight, against the
    # oracle's definition of the mode
    from rl_post_token_gb300 import _lib
    from tests.test_aggregate_weights import _check
    cfg, row_len, row_valid = case
    plan = _lib.grpo_plan_microbatches(cfg, np.asarray(row_len), np.asarray(row_valid))
    _check(plan, np.asarray(row_len, np.int64), np.asarray(row_valid, np.int64), agg)


@settings(**SETTINGS)
@given(st.one_of(fixed_or_dynamic(), compaction()))
def test_token_index_follows_its_definition(grpo_lib, case):
    # grpo_plan_token_index: exec token k of exec row j is token k of input row row_src[j],
    # stored as -1 - i for a padding row; checked on every plan the planner accepts
    from rl_post_token_gb300 import _lib
    cfg, row_len, third = case
    seg = third if cfg.get("compaction") else None
    valid = np.asarray(row_len) if seg is not None else np.asarray(third)
    try:
        p = _lib.grpo_plan_microbatches(cfg, np.asarray(row_len), valid, seg_counts=seg)
    except _lib.GrpoError:
        return
    rl = np.asarray(row_len, np.int64)
    off = np.concatenate([[0], np.cumsum(rl)])
    want = []
    for j in range(int(p["n_rows"])):
        r = int(p["row_src"][j])
        toks = list(range(int(off[r]), int(off[r + 1])))
        want += [-1 - t for t in toks] if p["row_pad"][j] else toks
    got = _lib.grpo_plan_token_index(p, rl)
    assert got.tolist() == want
