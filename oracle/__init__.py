"""Float64 CPU oracle for the GRPO/PPO policy-loss hot path.

THIS PACKAGE IS TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it. The product (the C-ABI library under
``rl_post_token_gb300``) never imports, links or calls it, and this package imports nothing
from the product: the two share no code, no constants and no helpers. Both sides are fed the
same seeded inputs by ``rl_post_token_gb300.workloads``, a generator module that holds none of
the method's arithmetic.

What it computes, each step written out plainly from the pages (see each module's docstring):

* ``oracle.planner``   -- how one collected batch becomes ``n_mini`` optimizer steps of
  forward/backward chunks: fixed chunks, context-compaction padding to a multiple of Q, and
  token-budget dynamic bins with order-restoring indices (integer only).
* ``oracle.advantage`` -- the group-normalised scalar advantage per rollout (float64).
* ``oracle.loss``      -- per-token log-softmax, ratio against the frozen pi_old, clipped
  surrogate, masking, the token-mean over the whole step and the analytic dlogits (float64).
* ``oracle.aggregate`` -- the step loss under token-mean and the two sequence-level modes,
  and the per-token gradient scale each implies (float64).

Pinning status (what ties each function to something other than itself; see ``tests/``):

* planner, fixed mode       -- the pages' 2x2 worked example and the 0/0 collapse (golden files).
* planner, compaction mode  -- the 4/8/4 = 16 rows, 3 pad rows example and its GPU table.
* planner, dynamic mode     -- invariants only (bin capacity, bin count bound, permutation,
  restore-after-permute is the identity). The particular binning rule is a reading of pages
  that name no algorithm: PARITY UNPINNED beyond those invariants.
* advantage                 -- hand-worked cases and numpy's own mean/std.
* loss / gradient           -- ratio == 1 closed form, scipy log_softmax, central finite
  differences on tiny vocabularies, row sums of dlogits, clip hand cases, padding rows.
* aggregation modes         -- a hand-worked step, closed forms relating the modes (equal
  full rows, a single row), linearity, central differences through the logits, row-order
  invariance, the empty step.
"""
