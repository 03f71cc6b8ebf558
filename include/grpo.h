/*
 * grpo.h -- C ABI of the GB300 (sm_103a) GRPO/PPO policy-loss hot path.
 *
 * One collected batch of rollouts is consumed as n_mini optimizer steps of n_micro
 * forward/backward chunks each, and every step's token-mean loss is divided once by N, the
 * number of valid (response_mask = 1) completion tokens of the whole step
 * ("Sizing mini-batches and micro-batches", sections "The core idea" and
 * "The hard part: deferred normalization").
 *
 * Typical step, all on one CUDA stream:
 *   grpo_plan_microbatches     host: which rows form which chunk and optimizer step, N per step
 *   grpo_group_advantage       device: group-normalised advantage per rollout, broadcast to tokens
 *   grpo_logprob_loss_fwd_bwd  device: per chunk, log-softmax + clipped surrogate + dlogits
 *   grpo_finish_step           device: the step's loss sum / max(N,1), metrics, deferred scaling
 *
 * Conventions shared by every entry point:
 *   - Status: every function returns int: GRPO_OK (0), a positive step status, or a negative
 *     GRPO_ERR_* code. No function aborts or prints.
 *   - Ownership: every buffer belongs to the caller, and the library never frees caller
 *     memory. The library allocates no device memory of its own with one exception: the
 *     module's 16 MiB device array of grpo_lmhead_forward_noalloc, held by every GPU that
 *     loads the library. The LM-head backward keeps one stream and four events per device
 *     (created on first use, kept until exit).
 *     "device" pointers are CUDA device memory of the current device; "host" pointers are
 *     ordinary host memory.
 *   - Asynchrony: device work is enqueued on `stream` (cudaStream_t passed as void*; NULL is
 *     the legacy default stream). Only grpo_finish_step with a non-NULL host result waits, so
 *     a whole step can be captured into a CUDA graph (after one call per kernel and
 *     shared-memory size has set the kernels' attributes).
 *   - Determinism: results depend only on the inputs, never on the chunking, the launch
 *     shape or the scheduling (no order-dependent floating-point atomics).
 *   - Environment switches (read on every call; for A/B comparison and tests; none changes a
 *     result bit, each only selects another instance of the same computation):
 *       GRPO_ROWPASS=c3|c4|l2     row pass: pin the 3- or 4-CTA cluster instance (bf16, where it
 *                                 fits) or the L2-streaming instance instead of the default
 *                                 2-CTA cluster;
 *       GRPO_ROWPASS_SLOTS=n      row pass: n shared-memory slices per CTA (0 = one fixed buffer
 *                                 per slice) where they fit, instead of as many as fit;
 *       GRPO_ROWPASS_FWD=0        forward-only calls take the general cluster kernel instead of
 *                                 the streaming forward kernel;
 *       GRPO_LMHEAD_CTA_GROUP=1   fused LM-head: one-CTA 128 x 256 tiles instead of paired
 *                                 2-CTA 256 x 256 tiles;
 *       GRPO_LMHEAD_OVERLAP=0     fused LM-head: the backward's launches all on the caller's
 *                                 stream instead of two streams.
 */
#ifndef GRPO_H_
#define GRPO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GRPO_API __attribute__((visibility("default")))
#else
#define GRPO_API
#endif

/* ---- status codes ---------------------------------------------------------------------- */
#define GRPO_OK                      0
#define GRPO_STEP_SKIPPED_NONFINITE  1   /* a valid token's log-prob or loss was not finite */
#define GRPO_ERR_INVALID            (-1) /* NULL pointer where one is required, bad size */
#define GRPO_ERR_DIVISIBILITY       (-2) /* batch % group_size, batch % mini, mini % micro */
#define GRPO_ERR_ROLLOUT_COUNT      (-3) /* the step does not hold exactly `batch` rollouts */
#define GRPO_ERR_TOKEN_BUDGET       (-4) /* a row is longer than max_token_len */
#define GRPO_ERR_INCOMPATIBLE       (-5) /* compaction with dynamic bins, packing, ... */
#define GRPO_ERR_CAPACITY           (-6) /* output arrays too small; sizes written back */
#define GRPO_ERR_CUDA               (-7) /* a CUDA runtime call failed */
#define GRPO_ERR_N_MISMATCH         (-8) /* counted N differs from the planner's N */
#define GRPO_ERR_KERNEL             (-9) /* a bounded wait inside a kernel gave up */
#define GRPO_ERR_UNSUPPORTED       (-10) /* dtype or device the library was not built for */

#define GRPO_DTYPE_F32   0
#define GRPO_DTYPE_BF16  1

#define GRPO_WORKLOAD_TOKENS     0  /* bin workload w = L       */
#define GRPO_WORKLOAD_ATTENTION  1  /* bin workload w = L * L   */

/* ---- planner ----------------------------------------------------------------------------- */

/* Planner configuration. Field meanings follow
 *  - "Sizing mini-batches and micro-batches", "The config surface": batch (trajectories per
 *    replica, a positive multiple of group_size), mini (per optimizer step, 0 = whole batch),
 *    micro (per forward/backward, 0 = one chunk); exact divisibility at every level;
 *  - "22-mini-batch-micro-batch-dynamic-batch-size的区别", section 3: dynamic token-budget bins
 *    (max_token_len, workload estimate, bins synced to a minimum count / rounded to a
 *    multiple, small bins at both ends);
 *  - "How a context-compaction step fits a variable number of rows into one batch":
 *    compaction pads each group to a multiple of Q = n_gpus * lcm(micro, logprob_batch) and
 *    rejects sequence packing, dynamic batching and the interleaved pipeline. */
typedef struct grpo_plan_cfg {
  int32_t batch;                 /* rollouts per replica per loop step (> 0) */
  int32_t mini;                  /* rollouts per optimizer step; 0 = batch */
  int32_t micro;                 /* rollouts (compaction: rows) per chunk; 0 = mini */
  int32_t group_size;            /* rollouts per prompt group (> 0) */
  int32_t dynamic;               /* 1 = token-budget bins inside each mini-batch */
  int32_t workload;              /* GRPO_WORKLOAD_* */
  int64_t max_token_len;         /* dynamic: token budget per bin (> 0) */
  int32_t min_bins;              /* dynamic: lower bound on bins per mini-batch */
  int32_t bin_multiple;          /* dynamic: bins per mini-batch rounded up to this (>= 1) */
  int32_t balance_ends;          /* dynamic: 1 = smallest bins at both ends */
  int32_t compaction;            /* 1 = context compaction */
  int32_t n_gpus;                /* compaction: GPUs the group is split across */
  int32_t logprob_batch;         /* compaction: log-prob micro batch */
  int32_t sequence_packing;      /* only checked against compaction */
  int32_t interleaved_pipeline;  /* only checked against compaction */
  int32_t use_rollout_logprobs;  /* 1 = rollout log-probs serve as pi_old */
} grpo_plan_cfg;

/* Plan of one collected batch. "Exec rows" are the rows in execution order (compaction adds
 * padding rows). Arrays are caller-owned HOST memory sized by the cap_* fields; on
 * GRPO_ERR_CAPACITY the scalar fields hold the required sizes and no array is written. */
typedef struct grpo_plan {
  int32_t cap_rows, cap_chunks, cap_steps;       /* in: capacities of the arrays below */
  int32_t n_rows;                /* out: exec rows */
  int32_t n_chunks;              /* out: forward/backward calls */
  int32_t n_steps;               /* out: optimizer steps (n_mini) */
  int32_t n_micro;               /* out: chunks per step if constant, else 0 (dynamic) */
  int32_t q;                     /* out: compaction multiple Q, else 0 */
  int32_t n_pad_rows;            /* out: padding rows (compaction) */
  int32_t needs_old_logp_cache;  /* out: n_steps > 1 and !use_rollout_logprobs */
  int32_t* row_src;              /* [cap_rows] input row feeding each exec row */
  int32_t* row_pad;              /* [cap_rows] 1 = padding row (mask 0, reward 0) */
  int32_t* row_gpu;              /* [cap_rows] GPU slot (compaction), else 0 */
  int32_t* row_rollout;          /* [cap_rows] rollout of the exec row, -1 for padding */
  int32_t* inv_perm;             /* [n_rows_in] exec position of each input row, or NULL */
  int32_t* chunk_row_off;        /* [cap_chunks + 1] exec-row offsets of the chunks */
  int32_t* step_chunk_off;       /* [cap_steps + 1] chunk offsets of the optimizer steps */
  int32_t* step_in_row_off;      /* [cap_steps + 1] input-row offsets of the steps */
  int64_t* chunk_tokens;         /* [cap_chunks] logits rows per chunk */
  int64_t* step_valid_tokens;    /* [cap_steps] N of each step */
  int32_t* step_valid_rows;      /* [cap_steps] rows with >= 1 valid token */
} grpo_plan;

/* Plan the (mini, micro) loop of one collected batch (host only, integer only).
 *  row_len[i]   logits rows (tokens) of input row i        host [n_rows_in]
 *  row_valid[i] mask = 1 positions of input row i          host [n_rows_in], 0 <= valid <= len
 *  seg_counts   rows produced by each rollout              host [n_rollouts], compaction only
 * Fixed mode: chunks of `micro` consecutive rows. Dynamic (inside each mini-batch):
 * k = max(ceil(sum L / max_token_len), min_bins, 1) rounded up to bin_multiple, capped at the
 * row count; rows visited by (workload desc, length desc, index asc) go to the feasible bin
 * (tokens + L <= max_token_len) with the least (workload, tokens, index), k growing to the
 * next multiple when none fits; rows by index inside a bin, bins by first row, or with
 * balance_ends the ascending (workload, first row) order dealt to positions 0, k-1, 1, ...
 * Compaction: each group padded to a multiple of Q with copies of its first real row.
 * Errors: GRPO_ERR_INVALID, _DIVISIBILITY, _ROLLOUT_COUNT, _TOKEN_BUDGET, _INCOMPATIBLE,
 * _CAPACITY. */
GRPO_API int grpo_plan_microbatches(const grpo_plan_cfg* cfg, int32_t n_rollouts,
                                    int32_t n_rows_in, const int32_t* row_len,
                                    const int32_t* row_valid, const int32_t* seg_counts,
                                    grpo_plan* out);

/* Expand a plan to one index per exec token (host only). For exec token t (exec rows in plan
 * order, tokens of a row consecutive) tok_src[t] is the input-order token it reads, or
 * -1 - that index for a padding row (masked: its logits row is still present, its loss is
 * 0). row_tok_off is the host [n_rows_in + 1] prefix sum of row_len. cap = length of
 * tok_src; the exec token count is written to *n_out (GRPO_ERR_CAPACITY if cap is short). */
GRPO_API int grpo_plan_token_index(const grpo_plan* plan, int32_t n_rows_in,
                                   const int64_t* row_tok_off, int64_t* tok_src, int64_t cap,
                                   int64_t* n_out);

/* Loss aggregation modes ("Sizing mini-batches and micro-batches", "The hard part: deferred
 * normalization": token mean over the step; "22-mini-batch-micro-batch-dynamic-batch-size的区别",
 * section 5: token-mean divides by the global token count, the sequence-level modes by the
 * global number of sequences). The pages do not print the sequence-level modes; reading, for
 * the input rows r of one step with n_r valid tokens, N = sum n_r and B = rows with n_r >= 1:
 *   TOKEN_MEAN          L = sum_t l_t / max(N, 1)
 *   SEQ_MEAN_TOKEN_SUM  L = sum_r (sum_{t in r} l_t) / max(B, 1)
 *   SEQ_MEAN_TOKEN_MEAN L = sum_r (sum_{t in r} l_t / max(n_r, 1)) / max(B, 1)
 * On one GPU the data-parallel compensation factor is 1. */
#define GRPO_AGG_TOKEN_MEAN          0
#define GRPO_AGG_SEQ_MEAN_TOKEN_SUM  1
#define GRPO_AGG_SEQ_MEAN_TOKEN_MEAN 2

/* Divisor, gradient scale and per-token weights of an aggregation mode for every optimizer step
 * of a plan (host only): step_divisor[s] = N_s (TOKEN_MEAN) or B_s (sequence-level modes);
 * when step_grad_scale is non-NULL, step_grad_scale[s] = 1/max(D_s, 1) (float64 division
 * rounded once to float: the grad_scale of the step's loss calls unless a deferred finish
 * applies it); when w_tok is non-NULL, w_tok[t] = 1/max(n_r, 1) rounded to float for every
 * token t of input row r under SEQ_MEAN_TOKEN_MEAN, else 1. A step's loss is then
 * sum_t w_t loss_t / max(D_s, 1) and each token's gradient scale grad_scale * w_t.
 *  plan            host, from grpo_plan_microbatches (step_in_row_off is read)
 *  row_tok_off     host int64 [n_rows_in + 1] token offsets of the input rows
 *  row_valid       host int32 [n_rows_in] mask = 1 positions per input row (as given to the planner)
 *  step_divisor    host int64 [plan->n_steps]
 *  w_tok           host float [row_tok_off[n_rows_in]] or NULL
 *  step_grad_scale host float [plan->n_steps] or NULL
 * Errors: GRPO_ERR_INVALID (NULL required pointer, unknown mode, inconsistent offsets). */
GRPO_API int grpo_plan_token_weights(const grpo_plan* plan, int32_t n_rows_in,
                                     const int64_t* row_tok_off, const int32_t* row_valid,
                                     int32_t agg, int64_t* step_divisor, float* w_tok,
                                     float* step_grad_scale);

/* ---- advantage --------------------------------------------------------------------------- */

/* Group-normalised advantage ("03 Data Protocol and Batch Lifecycle", response mask
 * semantics and reward/log-prob/advantage; "How a context-compaction step ...", why the row
 * count does not change the math, item 2). The pages print no formula; reading:
 *   A_r = (R_r - mean_g) / (std_g + eps), float64 inside, float32 out,
 * std unbiased (n-1) when unbiased_std != 0, groups = consecutive runs of group_size
 * rollouts, a single-rollout group (unbiased) or equal rewards give 0.
 *  rewards     device float [n_rollouts]
 *  adv_out     device float [n_rollouts]
 * Optional token broadcast (skipped when adv_tok is NULL):
 *  row_rollout device int32 [n_rows] rollout of each input row (-1 = padding -> 0), or NULL
 *              for row i = rollout i
 *  row_tok_off device int64 [n_rows + 1] token offsets of the rows
 *  adv_tok     device float [row_tok_off[n_rows]] */
GRPO_API int grpo_group_advantage(const float* rewards, int32_t n_rollouts, int32_t group_size,
                                  float eps, int32_t unbiased_std, float* adv_out,
                                  const int32_t* row_rollout, const int64_t* row_tok_off,
                                  int32_t n_rows, float* adv_tok, void* stream);

/* ---- loss forward + backward ------------------------------------------------------------- */

/* Device-resident step accumulator (caller-allocated, 128 bytes, zeroed once before the first
 * chunk). Loss calls add integer counts to it (order-independent); grpo_finish_step reads
 * them, writes `result`, and zeroes the counters for the next step. */
typedef struct grpo_step_result {
  double  loss;        /* loss_sum / max(D, 1), D the step's divisor (N unless the finish was
                          given another, see grpo_finish_step_ex) */
  double  loss_sum;    /* sum of loss_tok (times w_tok when given) over the step, float64,
                          fixed order */
  double  clipfrac;    /* n_clipped / max(N, 1) */
  int64_t n_valid;     /* N: mask = 1 tokens seen by the step's loss calls */
  int64_t n_clipped;   /* valid tokens whose clip bound (gradient 0) */
  int64_t n_nonfinite; /* valid tokens with a non-finite log-prob or loss */
  int64_t n_tokens;    /* logits rows processed */
  int32_t status;      /* GRPO_OK, GRPO_STEP_SKIPPED_NONFINITE, GRPO_ERR_N_MISMATCH, _KERNEL */
  int32_t kernel_flags;/* internal error bits (0 when healthy) */
} grpo_step_result;

typedef struct grpo_step_acc {
  uint64_t n_valid, n_clipped, n_nonfinite, n_tokens;
  uint32_t flags, reserved0;
  int64_t  divisor;     /* written by the finish: the step's divisor D (read by its gradient scaling) */
  uint64_t reserved[2];
  grpo_step_result result;
} grpo_step_acc;

/* One chunk of the step: per token row t of `logits`
 * ("Sizing mini-batches and micro-batches", "The problem", "The hard part: deferred
 * normalization", "pi_old must be frozen across the window"; the pages name an epsilon
 * clip without printing it, read here as the standard symmetric PPO clip):
 *   LSE = log sum_v exp(z_v); logp = z_y - LSE; r = exp(logp - old) (1 if old_logp NULL)
 *   loss_t = m * -min(r*A, clip(r, 1-eps, 1+eps)*A)
 *   dlogits_t = grad_scale * m * A * r * g * (softmax(z) - onehot(y)),
 *   g = 0 iff (A > 0 and r > 1+eps) or (A < 0 and r < 1-eps).
 * grad_scale is 1/max(N,1) with N from the planner (then chunked == un-chunked bit for bit),
 * or 1 with grpo_finish_step(deferred = 1) applying 1/max(N,1) once.
 *  logits    device [T, ld] GRPO_DTYPE_F32 or _BF16, row-major, V <= ld
 *  tok_src   device int64 [T] or NULL: side-input/output index of logits row t; negative
 *            (-1 - i) marks a padding row (mask 0). NULL means row t <-> index t.
 *  target    device int32, old_logp device float (or NULL), adv_tok device float,
 *  mask      device uint8: all indexed through tok_src
 *  dlogits   device [T, ld_out], same dtype as logits, or NULL (forward only: the pi_old
 *            ahead pass); masked rows are written as zeros
 *  loss_tok, logp_tok  device float, indexed through tok_src (logp_tok may be NULL); masked
 *            tokens get 0 in both
 *  acc       device grpo_step_acc
 * A target outside [0, V) makes that token's log-prob NaN (counted as non-finite).
 * Numerical range: the log-prob is formed as (z_y - shift) - log(sum), without cancellation.
 * Results are vouched for while the row's |LSE| <= 4096 (natural units; trained models' logits
 * are in the tens). A row beyond that reports a NaN log-prob and counts as non-finite, so the
 * step is skipped, instead of returning dlogits or an entropy degraded by the rounding at
 * that scale.
 * Errors: GRPO_ERR_INVALID (NULL required pointer, T < 0, V < 1, ld < V, T or V above
 * 2^31 - 1), GRPO_ERR_UNSUPPORTED (dtype), GRPO_ERR_CUDA (launch failure). */
GRPO_API int grpo_logprob_loss_fwd_bwd(const void* logits, int32_t dtype, int64_t T, int64_t V,
                                       int64_t ld, const int64_t* tok_src,
                                       const int32_t* target, const float* old_logp,
                                       const float* adv_tok, const uint8_t* mask,
                                       float clip_eps, float grad_scale, void* dlogits,
                                       int64_t ld_out, float* loss_tok, float* logp_tok,
                                       grpo_step_acc* acc, void* stream);

/* Regularisers that go through the same token-mean aggregation as the surrogate
 * ("22-mini-batch-micro-batch-dynamic-batch-size的区别", section 5: the entropy and KL losses
 * take the same global token count; "03 Data Protocol and Batch Lifecycle": the reference
 * policy's log-prob ref_log_prob). The pages give no formulas; the usual ones are used:
 *   + kl_coef * k,  k1 = logp - ref,  k3 = exp(ref - logp) - (ref - logp) - 1
 *   - ent_coef * H, H = -sum_v p_v log p_v  (an entropy bonus)
 * with gradients dk/dz = (dk/dlogp)(onehot - p) and dH/dz_v = -p_v (z_v - sum_u p_u z_u). */
#define GRPO_KL_NONE 0
#define GRPO_KL_K1   1
#define GRPO_KL_K3   2

typedef struct grpo_loss_terms {
  int32_t kl_kind;       /* GRPO_KL_* */
  float   kl_coef;
  const float* ref_logp; /* device float per token, indexed like old_logp; required for KL */
  float   ent_coef;      /* entropy bonus coefficient, 0 = off */
  float*  entropy_tok;   /* device float per token, indexed like loss_tok, or NULL; written
                            whenever non-NULL, also with ent_coef = 0 (entropy as a metric) */
  const float* w_tok;    /* device float per token, indexed like adv_tok, or NULL: a weight
                            multiplying grad_scale in that token's gradient (all terms), e.g.
                            1/max(n_r, 1) of GRPO_AGG_SEQ_MEAN_TOKEN_MEAN (see
                            grpo_plan_token_weights); loss_tok stays unweighted */
} grpo_loss_terms;

/* grpo_logprob_loss_fwd_bwd with the regularisers above added to every valid token's loss
 * and gradient (terms NULL: identical to grpo_logprob_loss_fwd_bwd). Masked tokens get 0 in
 * entropy_tok. Errors as grpo_logprob_loss_fwd_bwd, plus GRPO_ERR_INVALID for an unknown
 * kl_kind or a KL without ref_logp. */
GRPO_API int grpo_logprob_loss_fwd_bwd_ex(const void* logits, int32_t dtype, int64_t T, int64_t V,
                                          int64_t ld, const int64_t* tok_src,
                                          const int32_t* target, const float* old_logp,
                                          const float* adv_tok, const uint8_t* mask,
                                          float clip_eps, float grad_scale, void* dlogits,
                                          int64_t ld_out, float* loss_tok, float* logp_tok,
                                          const grpo_loss_terms* terms, grpo_step_acc* acc,
                                          void* stream);

/* grpo_logprob_loss_fwd_bwd_ex over logits that live in HOST memory (the page's problem: the
 * [T, V] logits of a step are many gigabytes; this streams them through a small device
 * buffer). Row t of the call is host row t (`ld` elements apart, `dtype` as above); every
 * other argument (side arrays, dlogits, outputs, terms, acc) is as in
 * grpo_logprob_loss_fwd_bwd_ex, on the device.
 * The rows go up in blocks of `block_rows`:
 *  - each block is copied into one half of `staging` on `copy_stream` (one cudaMemcpyAsync);
 *  - its row pass runs on `stream` once that copy has landed;
 *  - the next block's copy goes into the other half, so copy and row pass overlap.
 * The results are the bits grpo_logprob_loss_fwd_bwd_ex gives on the same rows in device
 * memory: a row's arithmetic does not depend on how the rows are split.
 * `staging`: device, 16-byte aligned, at least 2 * block_rows * ld * element-size bytes,
 * caller-owned. `logits_host`: pinned memory gives the link's full rate; pageable memory
 * works at a lower one. `copy_stream` may equal `stream` (no overlap).
 * Asynchronous: the first copy waits for the work already on `stream`, which may still read
 * `staging`. When `stream` has finished, all of the call's copies have too, and the host rows
 * may be reused.
 * Errors: as grpo_logprob_loss_fwd_bwd_ex; GRPO_ERR_INVALID also for a NULL host or staging
 * pointer, block_rows < 1 or misaligned staging; GRPO_ERR_CUDA for a failed copy or event call.
 * On an error after some blocks were enqueued, those blocks' work stays enqueued. */
GRPO_API int grpo_logprob_loss_fwd_bwd_host(const void* logits_host, int32_t dtype, int64_t T, int64_t V,
                                            int64_t ld, const int64_t* tok_src,
                                            const int32_t* target, const float* old_logp,
                                            const float* adv_tok, const uint8_t* mask,
                                            float clip_eps, float grad_scale, void* dlogits,
                                            int64_t ld_out, float* loss_tok, float* logp_tok,
                                            const grpo_loss_terms* terms, grpo_step_acc* acc,
                                            void* staging, int64_t block_rows, void* stream,
                                            void* copy_stream);

/* ---- step finish ------------------------------------------------------------------------- */

/* Close one optimizer step ("Sizing mini-batches and micro-batches", "The hard part:
 * deferred normalization", "Metric roll-up", "The poisoned-window countdown"):
 *   loss = sum(loss_tok[0..n_tok)) / max(N, 1) in float64 in a fixed order, N = counted
 *   valid tokens; counts are sums; if any valid token was non-finite the step is skipped:
 *   status GRPO_STEP_SKIPPED_NONFINITE and the registered gradient buffers are zeroed;
 *   otherwise, when deferred != 0, each buffer is scaled once by 1/max(N, 1) (scale, then
 *   the caller clips, then steps). expected_N >= 0 is checked against N
 *   (GRPO_ERR_N_MISMATCH in result.status).
 *  loss_tok    device float [n_tok]: the step's per-token losses (input order)
 *  grad_bufs   host array of n_bufs device pointers; grad_numels host int64 [n_bufs];
 *              grad_dtypes host int32 [n_bufs] (GRPO_DTYPE_*); may be NULL when n_bufs = 0
 *  result_host host grpo_step_result or NULL. If non-NULL the call copies acc->result to it,
 *              synchronises `stream` and returns result.status; if NULL it returns after
 *              enqueueing and the result stays in acc->result on the device.
 * Errors: GRPO_ERR_INVALID, GRPO_ERR_UNSUPPORTED, GRPO_ERR_CUDA. */
GRPO_API int grpo_finish_step(grpo_step_acc* acc, const float* loss_tok, int64_t n_tok,
                              int64_t expected_N, int32_t deferred, void* const* grad_bufs,
                              const int64_t* grad_numels, const int32_t* grad_dtypes,
                              int32_t n_bufs, grpo_step_result* result_host, void* stream);

/* grpo_finish_step for any aggregation mode: loss_sum = sum_t w_tok[t] * loss_tok[t] (each
 * product exact in float64; w_tok NULL = 1) in the same fixed order, loss = loss_sum /
 * max(D, 1) and the deferred gradient scale 1/max(D, 1), where D = divisor if >= 0, else the
 * counted N. grpo_finish_step is this call with w_tok NULL and divisor -1.
 *  w_tok    device float [n_tok] or NULL (the step's slice of grpo_plan_token_weights' output)
 * Data parallelism: when an optimizer step's rows are split across ranks, each rank runs its
 * rows with grad_scale = 1/max(D, 1) for the whole step's D (every rank can plan the whole
 * batch, so D needs no exchange) and finishes with divisor = D. The step's result is then the
 * sum over ranks of loss_sum and of the counts, with loss = that sum / max(D, 1); status is
 * the first error a rank reports, else skipped if any rank skipped. */
GRPO_API int grpo_finish_step_ex(grpo_step_acc* acc, const float* loss_tok, int64_t n_tok,
                                 const float* w_tok, int64_t divisor, int64_t expected_N,
                                 int32_t deferred, void* const* grad_bufs,
                                 const int64_t* grad_numels, const int32_t* grad_dtypes,
                                 int32_t n_bufs, grpo_step_result* result_host, void* stream);

/* ---- accumulation window (host) ----------------------------------------------------------- */

/* The trainer's view of one optimizer step fed chunk by chunk ("Sizing mini-batches and
 * micro-batches": "The hard part: deferred normalization", "The poisoned-window countdown",
 * "Metric roll-up"). Actions for each chunk: */
#define GRPO_WIN_ACCUMULATE 0  /* backprop the chunk and keep accumulating */
#define GRPO_WIN_STEP       1  /* backprop, scale the gradient by step_scale, clip, step */
#define GRPO_WIN_DISCARD    2  /* the chunk is non-finite: zero the gradients, window abandoned */
#define GRPO_WIN_DROP       3  /* a remaining chunk of an abandoned window: do not backprop */

typedef struct grpo_window {
  int32_t n_micro;            /* chunks per optimizer step */
  int32_t pos;                /* chunks of the current window seen */
  int32_t remaining_drop;     /* calls still to drop from an abandoned window */
  int32_t reserved0;
  int64_t denom;              /* divisors accumulated in the current window */
  double  loss_x_denom;       /* sum of chunk loss * chunk divisor in the current window */
  int64_t steps, skipped_windows, dropped_chunks;
  double  batch_loss_x_denom; /* roll-up over the trained windows */
  int64_t batch_denom;
} grpo_window;

/* Start a collected batch with n_micro >= 1 chunks per optimizer step (host only). */
GRPO_API int grpo_window_init(grpo_window* w, int32_t n_micro);

/* Feed one chunk: finite = 0 if its loss was non-finite; loss = the chunk's loss normalised
 * by its own divisor; denom = that divisor (valid tokens). Writes the action and, on
 * GRPO_WIN_STEP, step_scale = 1 / max(sum of the window's divisors, 1) (else 0). A
 * non-finite chunk discards its window and the window's remaining n_micro - pos chunks are
 * dropped before a fresh window starts; the divisor resets with it. */
GRPO_API int grpo_window_chunk(grpo_window* w, int32_t finite, double loss, int64_t denom,
                               int32_t* action, double* step_scale);

/* One optimizer step's result from the results of the n data-parallel ranks that ran its rows,
 * each rank's finish given the whole step's divisor (grpo_finish_step_ex) so that its gradients
 * already carry the step's one 1/max(D, 1) ("Sizing mini-batches and micro-batches", "The hard
 * part: deferred normalization"; "How a context-compaction step fits ...": the valid tokens are
 * summed over every GPU). Host only. The float64 loss sums and the counts are added in rank
 * order (index 0 first); loss = that sum / max(divisor, 1); clipfrac = n_clipped / max(n_valid,
 * 1); status = the first negative status in rank order, else GRPO_STEP_SKIPPED_NONFINITE if
 * any rank skipped, else GRPO_OK; kernel_flags are OR-ed.
 *  per_rank  host grpo_step_result [n] (the rank order is the summation order); n = 0 (per_rank
 *            may then be NULL) gives the empty step: every count and the loss 0, status OK
 *  divisor   the step's divisor D >= 0 (N for TOKEN_MEAN)
 *  out       host grpo_step_result (may alias none of per_rank)
 * Errors: GRPO_ERR_INVALID (NULL pointer, n < 0, divisor < 0). */
GRPO_API int grpo_combine_step_results(const grpo_step_result* per_rank, int32_t n, int64_t divisor,
                                       grpo_step_result* out);

/* Token-weighted loss sum(loss_i * denom_i) / max(sum(denom_i), 1) over the trained windows,
 * the summed divisor and the optimizer steps taken (any output may be NULL). */
GRPO_API int grpo_window_rollup(const grpo_window* w, double* loss, int64_t* denom, int64_t* steps);

/* ---- fused LM-head variant ---------------------------------------------------------------- */

/* Bytes of device workspace grpo_lmhead_loss_fwd_bwd needs for [T, H] hidden states and a
 * [V, H] output embedding: per-(token, 256-wide vocabulary tile) softmax partials (float32
 * shift and sum), per-token target logit, LSE and coefficient, two bf16 dlogits chunk
 * buffers [T, 256 * chunk_tiles], where the ceil(V/256) vocabulary tiles are split into
 * ceil(tiles/66) chunks of equal width (V = 151936: 9 chunks of 66 tiles, 16896 columns), and,
 * for the entropy bonus of grpo_lmhead_loss_fwd_bwd_ex, a third float32 partial per tile and
 * token and two float32 coefficients per token, then the backward's token partition (an int32
 * per token), its live count (one int32) and the live tokens' hidden states gathered into a
 * bf16 [T, H] buffer. Each part is rounded up to 256 bytes. 0 on bad sizes. */
GRPO_API size_t grpo_lmhead_workspace_size(int64_t T, int64_t V, int64_t H);

/* The same loss with the logits produced on the tensor cores: z = h W^T, computed tile by tile
 * and consumed by the softmax in the GEMM epilogue; no [T, V] matrix (logits, softmax,
 * exponentials or dlogits) is ever stored ("Sizing mini-batches and micro-batches", "The
 * problem"). All contractions are the library's own tcgen05 kernels (2-CTA clusters with
 * paired MMAs, 256 x 256 tiles, bf16 operands, float32 accumulation).
 *  - Forward: LSE, log-prob, ratio, clipped surrogate, per-token loss (as
 *    grpo_logprob_loss_fwd_bwd, one token per row of h).
 *  - Backward (d_h or dW non-NULL): over the live tokens only, those whose dlogits row is not
 *    all zero (a nonzero gradient coefficient, or with the entropy bonus a nonzero entropy
 *    term; a masked, clipped or zero-advantage token without regularisers has a zero row and
 *    its d_h row is written as zeros). Their hidden states are gathered in token order into the
 *    workspace; the live count stays on the device (no host synchronisation). Per vocabulary
 *    chunk, the chunk's logits of the live tokens are recomputed and their bf16 dlogits written
 *    to one of the two workspace chunk buffers; then d_h (+)= dlogits W_c, accumulated over the
 *    chunks in chunk order, and dW_c = dlogits^T h. The recompute makes the step
 *    2 T V H + 6 T_live V H flops (T_live = T when every token has a gradient). d_h and dW
 *    run on a second stream of the library's (one per device, created by the first call that
 *    needs it, which should come before any stream capture), so the next chunk's recompute
 *    runs beside them; the call's work on both streams is done when `stream` reaches the
 *    call's end.
 *  - Determinism: d_h and the per-token outputs of a token do not depend on which other
 *    tokens share the call; dW sums over the call's tokens in a fixed order.
 *  h          device bf16 [T, H] row-major, 16-byte aligned; H a multiple of 64
 *  W          device bf16 [V, H] row-major, 16-byte aligned
 *  target, old_logp (or NULL), adv_tok, mask   device, indexed by token row
 *  grad_scale 1/max(N,1) (or 1 with a deferred finish on d_h / dW)
 *  d_h        device float [T, H] or NULL; dW device float [V, H] or NULL (both NULL: forward
 *             only); each 16-byte aligned
 *  flags      0: dW = dlogits^T h of this call's tokens; GRPO_LMHEAD_DW_ACCUMULATE: dW += it, so
 *             the micro-batches of one optimizer step (one call each, grad_scale the step's
 *             1/max(N,1), or 1 with a deferred finish over d_h and dW) sum into one dW, each
 *             call's float32 product added in call order ("Sizing mini-batches and
 *             micro-batches", "The hard part: deferred normalization": the chunks' gradients
 *             sum to the un-chunked step's). d_h rows and per-token outputs never accumulate.
 *             GRPO_LMHEAD_SKIP_MASKED: pass A skips the masked tokens (same results).
 *             Other bits: GRPO_ERR_INVALID.
 *  loss_tok, logp_tok (or NULL)  device float [T]
 *  acc        device grpo_step_acc (counts as in grpo_logprob_loss_fwd_bwd)
 *  workspace  device, 256-byte aligned, >= grpo_lmhead_workspace_size(T, V, H) bytes,
 *             caller-owned; it holds all of the call's scratch, so calls may overlap (several
 *             streams, several host threads) as long as each has its own workspace and outputs
 * Environment: GRPO_LMHEAD_CTA_GROUP=1 selects one-CTA 128 x 256 tiles instead of the paired
 * 256 x 256 tiles; GRPO_LMHEAD_OVERLAP=0 keeps every launch on `stream` (same results).
 * Errors: GRPO_ERR_INVALID (sizes, NULL, alignment), GRPO_ERR_CAPACITY (workspace too small),
 * GRPO_ERR_UNSUPPORTED (tensor-map creation), GRPO_ERR_CUDA. */
#define GRPO_LMHEAD_DW_ACCUMULATE 1u /* flags: dW += dlogits^T h (the call's tokens added to dW) */
/* flags: pass A (the forward GEMM) runs over the mask=1 tokens only. They are put first in a
 * stable compact order (the count stays on the device) and their hidden states gathered into
 * the workspace. That costs one partition and one gather (about 40 us at 16384 tokens) and
 * saves the forward GEMM's work for every masked token, e.g. padding rows. The results are
 * the same bits as without the flag. */
#define GRPO_LMHEAD_SKIP_MASKED 2u

GRPO_API int grpo_lmhead_loss_fwd_bwd(const void* h, const void* W, int64_t T, int64_t V, int64_t H,
                                      const int32_t* target, const float* old_logp,
                                      const float* adv_tok, const uint8_t* mask, float clip_eps,
                                      float grad_scale, float* d_h, float* dW, uint32_t flags,
                                      float* loss_tok, float* logp_tok, grpo_step_acc* acc,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* grpo_lmhead_loss_fwd_bwd with the regularisers of grpo_loss_terms added to every valid
 * token's loss and gradient, as grpo_logprob_loss_fwd_bwd_ex adds them to the row pass (terms
 * NULL: identical to grpo_lmhead_loss_fwd_bwd). KL to the reference policy (k1 or k3) and the
 * per-token weight w_tok act on each token's gradient coefficient. The entropy bonus (ent_coef,
 * or an entropy_tok output) makes pass A carry sum e z per vocabulary tile as well, and, with
 * ent_coef != 0, the backward's dlogits take the form p_v (a + b z_v) - coef [v == y]
 * (b = ent_coef * grad_scale * w, a = coef - b E_p[z]), so the bonus's gradient reaches d_h and
 * dW. loss_tok stays unweighted; entropy_tok (natural units) is written for every token,
 * 0 for masked ones. Indices: ref_logp and w_tok as adv_tok, entropy_tok as loss_tok.
 * Errors: those of grpo_lmhead_loss_fwd_bwd, and GRPO_ERR_INVALID for an unknown kl_kind, a KL
 * term without ref_logp, or a non-finite coefficient. */
GRPO_API int grpo_lmhead_loss_fwd_bwd_ex(const void* h, const void* W, int64_t T, int64_t V, int64_t H,
                                         const int32_t* target, const float* old_logp,
                                         const float* adv_tok, const uint8_t* mask, float clip_eps,
                                         float grad_scale, float* d_h, float* dW, uint32_t flags,
                                         float* loss_tok, float* logp_tok, const grpo_loss_terms* terms,
                                         grpo_step_acc* acc, void* workspace, size_t workspace_bytes,
                                         void* stream);

/* Allocation-free forward pass of the fused LM-head variant. The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory when they need the
 * loss -- a serving or scoring process whose device memory is all handed to its own pool (a
 * KV cache or caching allocator), where a new cudaMalloc would fail or force the pool to
 * shrink, or a code path that must not risk the device synchronisation cudaMalloc/cudaFree
 * can cause. It computes what grpo_lmhead_loss_fwd_bwd computes with d_h = dW = NULL
 * (per-token loss and log-prob, counts in acc) and calls no cudaMalloc, cudaFree or
 * allocating library routine.
 *  - Its scratch is a 16 MiB file-scope device array inside this library
 *    (grpo_lmhead_forward_noalloc_max_scratch() bytes); every GPU that loads the library holds
 *    it until the process exits.
 *  - Limit: 4*T*(2*ceil(V/256) + 3) bytes (each part rounded up to 256) must fit the array,
 *    e.g. about 3,500 tokens at V = 151936; larger calls return GRPO_ERR_CAPACITY and launch
 *    nothing.
 *  - The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 *    with that device current) and sets the GEMM kernel's shared-memory limit; make that first
 *    call before any stream capture. The address is kept with the id of the device's context:
 *    if that context is destroyed and re-created (cudaDeviceReset), the next call looks the
 *    address up again, so the same rule applies to it.
 *  - Every call shares the one array and leaves its contents behind; no part of it needs to
 *    start at zero (each location a call reads was written earlier in that call), but calls
 *    that overlap on the GPU (several streams, several host threads) race: serialise them.
 * Arguments, layouts and other errors as grpo_lmhead_loss_fwd_bwd. */
GRPO_API int grpo_lmhead_forward_noalloc(const void* h, const void* W, int64_t T, int64_t V, int64_t H,
                                         const int32_t* target, const float* old_logp,
                                         const float* adv_tok, const uint8_t* mask, float clip_eps,
                                         float grad_scale, float* loss_tok, float* logp_tok,
                                         grpo_step_acc* acc, void* stream);

/* Size in bytes of grpo_lmhead_forward_noalloc's scratch array. */
GRPO_API size_t grpo_lmhead_forward_noalloc_max_scratch(void);

/* ---- misc -------------------------------------------------------------------------------- */

/* Static string naming a status code. */
GRPO_API const char* grpo_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
GRPO_API int grpo_version(void);

/* Self-test of the bounded waits every pipelined kernel of this library relies on (no page
 * defines it). Launches one CTA on `stream` that waits on an mbarrier nothing completes. The wait
 * gives up after its limit, the same one the row-pass and LM-head kernels use: about one
 * second, or 2^24 polls if those end sooner. The kernel then raises the wait-timeout bit of
 * acc->flags, as a kernel whose pipeline broke would. The next grpo_finish_step on `acc`
 * reports GRPO_ERR_KERNEL and zeroes the gradient buffers it is given.
 * `acc`: device pointer to a caller-owned accumulator. Returns GRPO_ERR_INVALID for a NULL
 * `acc`, GRPO_ERR_CUDA if the launch fails, else GRPO_OK (asynchronous). */
GRPO_API int grpo_selftest_wait_timeout(grpo_step_acc* acc, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GRPO_H_ */
