"""Oracle of the trainer's accumulation window: deferred normalisation, the poisoned-window
countdown and the token-weighted metric roll-up. Test infrastructure only; see
``oracle/__init__.py``.

Sources ("Sizing mini-batches and micro-batches"):
* *The hard part: deferred normalization*: each chunk reports its divisor; the trainer sums
  them over the window and, on the window's last chunk, scales the gradient once by
  1 / max(sum, 1), then clips, then steps.
* *The poisoned-window countdown*: a chunk whose loss is non-finite discards the current
  window (gradients zeroed, accumulator reset); the trainer remembers how many chunks of that
  window are still to come and drops exactly that many following calls before a fresh window
  starts; the divisor resets with it. With one chunk per window nothing is dropped.
* *Metric roll-up*: the logged loss of the collected batch is sum(loss_i * denom_i) /
  sum(denom_i) over the chunks that were trained (each chunk's loss is normalised by its own
  divisor); counts are sums, not averages.

Actions returned per chunk: ACCUMULATE (backprop, keep accumulating), STEP (backprop, then
scale by the returned factor, clip, step), DISCARD (non-finite: zero the gradients, the
window is abandoned), DROP (a remaining chunk of an abandoned window: do not backprop).
"""
from __future__ import annotations

ACCUMULATE, STEP, DISCARD, DROP = 0, 1, 2, 3


class Window:
    def __init__(self, n_micro: int):
        if n_micro < 1:
            raise ValueError("n_micro >= 1")
        self.n_micro = n_micro
        self.pos = 0              # chunks of the current window seen so far
        self.remaining_drop = 0   # calls still to drop from an abandoned window
        self.denom = 0            # divisors accumulated in the current window
        self.loss_x_denom = 0.0   # sum of chunk loss * chunk divisor in the current window
        self.steps = 0
        self.skipped_windows = 0
        self.dropped_chunks = 0
        self.batch_loss_x_denom = 0.0
        self.batch_denom = 0

    def chunk(self, finite: bool, loss: float, denom: int):
        """Returns (action, scale); scale = 1 / max(window divisor, 1) on STEP, else 0."""
        if self.remaining_drop > 0:
            self.remaining_drop -= 1
            self.dropped_chunks += 1
            return DROP, 0.0
        self.pos += 1
        if not finite:
            self.remaining_drop = self.n_micro - self.pos
            self.pos = 0
            self.denom = 0
            self.loss_x_denom = 0.0
            self.skipped_windows += 1
            return DISCARD, 0.0
        self.denom += int(denom)
        self.loss_x_denom += float(loss) * int(denom)
        if self.pos < self.n_micro:
            return ACCUMULATE, 0.0
        scale = 1.0 / max(self.denom, 1)
        self.batch_loss_x_denom += self.loss_x_denom
        self.batch_denom += self.denom
        self.steps += 1
        self.pos = 0
        self.denom = 0
        self.loss_x_denom = 0.0
        return STEP, scale

    def rollup(self):
        """(token-weighted loss of the trained windows, summed divisor, optimizer steps)."""
        return self.batch_loss_x_denom / max(self.batch_denom, 1), self.batch_denom, self.steps
