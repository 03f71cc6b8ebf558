"""Randomised search (hypothesis) for any plan on which the library's host planner and the
oracle planner disagree: every field and every error code, over fixed, dynamic and
compaction configurations. Host code only."""
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
