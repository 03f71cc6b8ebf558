// Host state machine of the trainer's accumulation window ("Sizing mini-batches and
// micro-batches": "The hard part: deferred normalization" -- divisors summed over the window,
// one 1/max(sum, 1) scale on its last chunk, then clip, then step; "The poisoned-window
// countdown" -- a non-finite chunk discards its window and exactly the window's remaining
// chunks are dropped before a fresh window starts, the divisor reset with it; "Metric
// roll-up" -- the batch loss is sum(loss_i * denom_i) / sum(denom_i) over the trained chunks,
// counts are sums).
#include <cmath>

#include "grpo.h"

extern "C" GRPO_API int grpo_window_init(grpo_window* w, int32_t n_micro) {
  if (!w || n_micro < 1) return GRPO_ERR_INVALID;
  *w = grpo_window{};
  w->n_micro = n_micro;
  return GRPO_OK;
}

extern "C" GRPO_API int grpo_window_chunk(grpo_window* w, int32_t finite, double loss, int64_t denom,
                                          int32_t* action, double* step_scale) {
  if (!w || !action || w->n_micro < 1 || denom < 0) return GRPO_ERR_INVALID;
  if (step_scale) *step_scale = 0.0;
  if (w->remaining_drop > 0) {  // a leftover chunk of an abandoned window
    --w->remaining_drop;
    ++w->dropped_chunks;
    *action = GRPO_WIN_DROP;
    return GRPO_OK;
  }
  ++w->pos;
  if (!finite) {
    w->remaining_drop = w->n_micro - w->pos;
    w->pos = 0;
    w->denom = 0;
    w->loss_x_denom = 0.0;
    ++w->skipped_windows;
    *action = GRPO_WIN_DISCARD;
    return GRPO_OK;
  }
  w->denom += denom;
  w->loss_x_denom += loss * (double)denom;
  if (w->pos < w->n_micro) {
    *action = GRPO_WIN_ACCUMULATE;
    return GRPO_OK;
  }
  if (step_scale) *step_scale = 1.0 / (double)(w->denom > 1 ? w->denom : 1);
  w->batch_loss_x_denom += w->loss_x_denom;
  w->batch_denom += w->denom;
  ++w->steps;
  w->pos = 0;
  w->denom = 0;
  w->loss_x_denom = 0.0;
  *action = GRPO_WIN_STEP;
  return GRPO_OK;
}

extern "C" GRPO_API int grpo_window_rollup(const grpo_window* w, double* loss, int64_t* denom, int64_t* steps) {
  if (!w) return GRPO_ERR_INVALID;
  if (loss) *loss = w->batch_loss_x_denom / (double)(w->batch_denom > 1 ? w->batch_denom : 1);
  if (denom) *denom = w->batch_denom;
  if (steps) *steps = w->steps;
  return GRPO_OK;
}

// One optimizer step's result from the results of the data-parallel ranks that ran its rows,
// each finished with the step's divisor D ("Sizing mini-batches and micro-batches", "The hard
// part: deferred normalization": the step's loss is divided once by the count of the whole
// step; "How a context-compaction step fits ...": the valid tokens are summed over every GPU).
// The float64 loss sums and the counts are added in rank order; loss = sum / max(D, 1).
extern "C" GRPO_API int grpo_combine_step_results(const grpo_step_result* per_rank, int32_t n, int64_t divisor,
                                                  grpo_step_result* out) {
  if ((!per_rank && n > 0) || !out || n < 0 || divisor < 0) return GRPO_ERR_INVALID;
  grpo_step_result r{};
  r.status = GRPO_OK;
  for (int32_t k = 0; k < n; ++k) {
    const grpo_step_result& x = per_rank[k];
    r.loss_sum += x.loss_sum;
    r.n_valid += x.n_valid;
    r.n_clipped += x.n_clipped;
    r.n_nonfinite += x.n_nonfinite;
    r.n_tokens += x.n_tokens;
    if (x.status < 0 && r.status >= 0)
      r.status = x.status;  // the first error, in rank order
    else if (x.status == GRPO_STEP_SKIPPED_NONFINITE && r.status == GRPO_OK)
      r.status = x.status;
    r.kernel_flags |= x.kernel_flags;
  }
  r.loss = r.loss_sum / (double)(divisor > 1 ? divisor : 1);
  r.clipfrac = (double)r.n_clipped / (double)(r.n_valid > 1 ? r.n_valid : 1);
  *out = r;
  return GRPO_OK;
}
