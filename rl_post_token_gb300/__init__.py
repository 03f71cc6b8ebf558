"""GB300-native GRPO/PPO policy-loss hot path.

The product is the C-ABI library ``libgrpo.so`` (declared in ``include/grpo.h``, sources in
``csrc/``); this package holds its in-tree build script (``build``), a thin ctypes binding with
the same entry-point names (``_lib``), and the seeded synthetic input generators
(``workloads``). Importing the package does not load the library; the first call does, and it
raises if the library has not been built.
"""
from ._lib import (  # noqa: F401
    GrpoError,
    grpo_finish_step,
    grpo_group_advantage,
    grpo_lmhead_loss_fwd_bwd,
    grpo_lmhead_workspace_size,
    grpo_logprob_loss_fwd_bwd,
    grpo_plan_microbatches,
    grpo_plan_token_index,
    grpo_version,
    lib,
    new_step_acc,
    read_step_result,
)
