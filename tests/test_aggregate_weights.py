"""The library's aggregation weights (grpo_plan_token_weights, host code) against the oracle's
definitions of each mode applied to every optimizer step of a plan. No GPU needed."""
import numpy as np
import pytest

from oracle import aggregate as AG
from rl_post_token_gb300 import workloads as W


def _prefix_mask(row_len, row_valid):
    return np.concatenate([np.r_[np.ones(v, np.uint8), np.zeros(L - v, np.uint8)]
                           for L, v in zip(row_len, row_valid)]) if len(row_len) else np.zeros(0, np.uint8)


def _check(plan, row_len, row_valid, agg):
    from rl_post_token_gb300 import _lib
    div, w = _lib.grpo_plan_token_weights(plan, row_len, row_valid, agg)
    div2, none, scale = _lib.grpo_plan_token_weights(plan, row_len, row_valid, agg, want_w=False, want_scale=True)
    assert none is None and np.array_equal(div2, div)
    off = np.concatenate([[0], np.cumsum(np.asarray(row_len, np.int64))])
    mask = _prefix_mask(row_len, row_valid)
    for s in range(plan["n_steps"]):
        r0, r1 = plan["step_in_row_off"][s], plan["step_in_row_off"][s + 1]
        soff = off[r0:r1 + 1] - off[r0]
        m = mask[off[r0]:off[r1]]
        assert div[s] == AG.divisor(soff, m, agg)
        # the step's gradient scale: the oracle's 1/max(D, 1), rounded once to float32
        assert scale[s] == np.float32(1.0 / max(AG.divisor(soff, m, agg), 1))
        # the weight is the oracle's per-token scale without the step's 1/max(D, 1)
        want = AG.token_scale(soff, m, agg) * max(AG.divisor(soff, m, agg), 1)
        np.testing.assert_allclose(w[off[r0]:off[r1]], want, rtol=1e-7, atol=0)
    if agg == AG.TOKEN_MEAN:
        assert np.array_equal(div, plan["step_valid_tokens"])
    else:
        assert np.array_equal(div, plan["step_valid_rows"])


@pytest.mark.parametrize("agg", [AG.TOKEN_MEAN, AG.SEQ_MEAN_TOKEN_SUM, AG.SEQ_MEAN_TOKEN_MEAN])
@pytest.mark.parametrize("name", ["tiny", "qwen_step", "dynamic", "compaction"])
def test_workload_weights(grpo_lib, name, agg):
    from rl_post_token_gb300 import _lib
    wl = W.make_workload(name, valid_lo=0) if name == "tiny" else W.make_workload(name)
    plan = _lib.grpo_plan_microbatches(wl.plan, wl.row_len, wl.row_valid, seg_counts=wl.seg_counts)
    _check(plan, wl.row_len, wl.row_valid, agg)


@pytest.mark.parametrize("seed", range(12))
def test_random_plans(grpo_lib, seed):
    from rl_post_token_gb300 import _lib
    rng = np.random.default_rng(100 + seed)
    B = 4 * int(rng.integers(1, 9))
    row_len = rng.integers(0, 40, B)
    row_valid = np.array([rng.integers(0, L + 1) for L in row_len])
    mini = B // int(rng.choice([d for d in (1, 2, 4) if B % d == 0]))
    cfg = dict(batch=B, mini=mini, micro=mini, group_size=4)
    plan = _lib.grpo_plan_microbatches(cfg, row_len, row_valid)
    for agg in (AG.TOKEN_MEAN, AG.SEQ_MEAN_TOKEN_SUM, AG.SEQ_MEAN_TOKEN_MEAN):
        _check(plan, row_len, row_valid, agg)


def test_errors(grpo_lib):
    from rl_post_token_gb300 import _lib
    wl = W.make_workload("tiny")
    plan = _lib.grpo_plan_microbatches(wl.plan, wl.row_len, wl.row_valid)
    with pytest.raises(_lib.GrpoError) as e:
        _lib.grpo_plan_token_weights(plan, wl.row_len, wl.row_valid, 3)
    assert e.value.code == _lib.ERR_INVALID
    bad = np.array(wl.row_valid)
    bad[0] = wl.row_len[0] + 1  # more valid positions than tokens
    with pytest.raises(_lib.GrpoError) as e:
        _lib.grpo_plan_token_weights(plan, wl.row_len, bad, 0)
    assert e.value.code == _lib.ERR_INVALID
