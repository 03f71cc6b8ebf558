// Host planner: one collected batch -> optimizer steps -> forward/backward chunks.
//
// Integer-only scheduling logic that runs on the host before any kernel:
//  * fixed chunks  ("Sizing mini-batches and micro-batches", "The config surface" and
//    "A worked example": n_mini = batch / mini, n_micro = mini / micro, 0 = one chunk,
//    exact divisibility at every level);
//  * dynamic token-budget bins inside each mini-batch ("22-mini-batch-micro-batch-dynamic-
//    batch-size的区别", section 3: every row fits the budget, the bin count is the token total
//    over the budget rounded up, rows are binned by an estimated workload, small bins may go
//    to both ends, an index map restores the order);
//  * context compaction ("How a context-compaction step fits a variable number of rows into
//    one batch": each group padded to a multiple of Q = n_gpus * lcm(micro, logprob_batch)
//    with masked copies of a real row, each group split evenly across GPUs in contiguous
//    blocks, exactly `batch` rollouts per step, one optimizer step).
// The dynamic rule is fully specified here because the pages name no algorithm:
//   k = max(ceil(total / budget), min_bins, 1) rounded up to bin_multiple, capped at the row
//   count; rows visited by (workload desc, length desc, index asc); each row goes to the
//   feasible bin (tokens + L <= budget) with the least (workload, tokens, index); if none is
//   feasible k grows to the next multiple and the binning restarts; rows sorted inside a bin;
//   bins ordered by smallest row, or, with balance_ends, the ascending (workload, smallest
//   row) order dealt to positions 0, k-1, 1, k-2, ...
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <limits>
#include <numeric>
#include <vector>

#include "grpo.h"

namespace {

struct PlanOut {
  std::vector<int32_t> row_src, row_pad, row_gpu, row_rollout;
  std::vector<int32_t> chunk_row_off{0}, step_chunk_off{0}, step_in_row_off{0};
  int32_t n_micro = 0, q = 0;
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t m) { return m > 1 ? ceil_div(a, m) * m : a; }

// Bins of one mini-batch: rows [r0, r1) in input order. Appends rows to out.row_src and one
// chunk offset per bin.
void dynamic_bins(const grpo_plan_cfg& c, int32_t r0, int32_t r1, const int32_t* len,
                  PlanOut& out) {
  const int64_t B = r1 - r0;
  const int64_t cap = c.max_token_len;
  int64_t total = 0;
  for (int32_t r = r0; r < r1; ++r) total += len[r];
  int64_t k = std::max<int64_t>({ceil_div(total, cap), (int64_t)c.min_bins, 1});
  k = std::min<int64_t>(round_up(k, c.bin_multiple), B);

  auto weight = [&](int32_t r) -> int64_t {
    const int64_t L = len[r];
    return c.workload == GRPO_WORKLOAD_ATTENTION ? L * L : L;
  };
  std::vector<int32_t> visit(B);
  std::iota(visit.begin(), visit.end(), r0);
  std::sort(visit.begin(), visit.end(), [&](int32_t a, int32_t b) {
    const int64_t wa = weight(a), wb = weight(b);
    if (wa != wb) return wa > wb;
    if (len[a] != len[b]) return len[a] > len[b];
    return a < b;
  });

  std::vector<int64_t> load_w, load_t;
  std::vector<std::vector<int32_t>> members;
  for (;;) {
    load_w.assign(k, 0);
    load_t.assign(k, 0);
    members.assign(k, {});
    bool feasible = true;
    for (int32_t r : visit) {
      int64_t best = -1;
      for (int64_t b = 0; b < k; ++b) {
        if (load_t[b] + len[r] > cap) continue;
        if (best < 0 || load_w[b] < load_w[best] ||
            (load_w[b] == load_w[best] && load_t[b] < load_t[best]))
          best = b;  // equal (workload, tokens): the lower index, found first, stays
      }
      if (best < 0) { feasible = false; break; }
      members[best].push_back(r);
      load_w[best] += weight(r);
      load_t[best] += len[r];
    }
    if (feasible) break;
    k = std::min<int64_t>(round_up(k + 1, c.bin_multiple), B);  // k == B always fits
  }

  constexpr int64_t kNone = std::numeric_limits<int64_t>::max();
  auto first = [&](int64_t b) -> int64_t { return members[b].empty() ? kNone : members[b][0]; };
  for (auto& m : members) std::sort(m.begin(), m.end());
  std::vector<int64_t> order(k);
  std::iota(order.begin(), order.end(), 0);
  std::sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
    return first(a) != first(b) ? first(a) < first(b) : a < b;
  });
  if (c.balance_ends) {
    std::vector<int64_t> asc(order);
    std::sort(asc.begin(), asc.end(), [&](int64_t a, int64_t b) {
      if (load_w[a] != load_w[b]) return load_w[a] < load_w[b];
      if (first(a) != first(b)) return first(a) < first(b);
      return a < b;
    });
    int64_t lo = 0, hi = k - 1;
    for (int64_t i = 0; i < k; ++i) order[(i % 2 == 0) ? lo++ : hi--] = asc[i];
  }
  for (int64_t b : order) {
    for (int32_t r : members[b]) out.row_src.push_back(r);
    out.chunk_row_off.push_back((int32_t)out.row_src.size());
  }
}

int plan_compaction(const grpo_plan_cfg& c, int32_t n_rollouts, int32_t n_rows_in,
                    const int32_t* seg, PlanOut& out) {
  if (c.dynamic || c.sequence_packing || c.interleaved_pipeline) return GRPO_ERR_INCOMPATIBLE;
  if (c.mini != 0 && c.mini != c.batch) return GRPO_ERR_INCOMPATIBLE;
  if (!seg || c.micro <= 0 || c.n_gpus <= 0 || c.logprob_batch <= 0) return GRPO_ERR_INVALID;
  int64_t rows = 0;
  for (int32_t r = 0; r < n_rollouts; ++r) {
    if (seg[r] < 1) return GRPO_ERR_INVALID;
    rows += seg[r];
  }
  if (rows != n_rows_in) return GRPO_ERR_INVALID;
  if (n_rollouts != c.batch) return GRPO_ERR_ROLLOUT_COUNT;

  const int64_t g = std::gcd<int64_t>(c.micro, c.logprob_batch);
  const int64_t Q = (int64_t)c.n_gpus * (c.micro / g * c.logprob_batch);
  if (Q > std::numeric_limits<int32_t>::max()) return GRPO_ERR_INVALID;
  out.q = (int32_t)Q;
  const int32_t G = c.group_size;
  int32_t row = 0;  // first input row of the current rollout
  for (int32_t g0 = 0; g0 < c.batch; g0 += G) {
    const int32_t first_row = row;
    int32_t real = 0;
    for (int32_t r = g0; r < g0 + G; ++r) {
      for (int32_t s = 0; s < seg[r]; ++s) {
        out.row_src.push_back(row + s);
        out.row_rollout.push_back(r);
        out.row_pad.push_back(0);
      }
      row += seg[r];
      real += seg[r];
    }
    const int64_t padded = ceil_div(real, Q) * Q;
    for (int64_t k = real; k < padded; ++k) {
      out.row_src.push_back(first_row);  // a padding row copies the group's first real row
      out.row_rollout.push_back(-1);
      out.row_pad.push_back(1);
    }
    const int64_t per_gpu = padded / c.n_gpus;
    for (int64_t k = 0; k < padded; ++k) out.row_gpu.push_back((int32_t)(k / per_gpu));
  }
  const int32_t n_exec = (int32_t)out.row_src.size();
  for (int32_t j = c.micro; j <= n_exec; j += c.micro) out.chunk_row_off.push_back(j);
  out.step_chunk_off.push_back((int32_t)out.chunk_row_off.size() - 1);
  out.step_in_row_off.push_back(n_rows_in);
  out.n_micro = (int32_t)out.chunk_row_off.size() - 1;
  return GRPO_OK;
}

}  // namespace

extern "C" GRPO_API int grpo_plan_microbatches(const grpo_plan_cfg* cfg, int32_t n_rollouts,
                                               int32_t n_rows_in, const int32_t* row_len,
                                               const int32_t* row_valid,
                                               const int32_t* seg_counts, grpo_plan* out) {
  if (!cfg || !out || n_rows_in < 0 || n_rollouts < 0) return GRPO_ERR_INVALID;
  if (n_rows_in > 0 && (!row_len || !row_valid)) return GRPO_ERR_INVALID;
  const grpo_plan_cfg& c = *cfg;
  for (int32_t i = 0; i < n_rows_in; ++i)
    if (row_len[i] < 0 || row_valid[i] < 0 || row_valid[i] > row_len[i]) return GRPO_ERR_INVALID;
  if (c.batch <= 0 || c.group_size <= 0 || c.mini < 0 || c.micro < 0) return GRPO_ERR_INVALID;
  if (c.batch % c.group_size != 0) return GRPO_ERR_DIVISIBILITY;

  PlanOut p;
  int32_t n_steps = 0;
  if (c.compaction) {
    const int rc = plan_compaction(c, n_rollouts, n_rows_in, seg_counts, p);
    if (rc != GRPO_OK) return rc;
    n_steps = 1;
  } else {
    if (n_rollouts != c.batch || n_rows_in != c.batch) return GRPO_ERR_ROLLOUT_COUNT;
    const int32_t mini = c.mini ? c.mini : c.batch;
    const int32_t micro = c.micro ? c.micro : mini;
    if (c.batch % mini != 0 || mini % micro != 0) return GRPO_ERR_DIVISIBILITY;
    n_steps = c.batch / mini;
    for (int32_t i = 1; i <= n_steps; ++i) p.step_in_row_off.push_back(i * mini);
    if (!c.dynamic) {
      p.n_micro = mini / micro;
      p.row_src.resize(c.batch);
      std::iota(p.row_src.begin(), p.row_src.end(), 0);
      for (int32_t j = micro; j <= c.batch; j += micro) p.chunk_row_off.push_back(j);
      for (int32_t i = 1; i <= n_steps; ++i) p.step_chunk_off.push_back(i * p.n_micro);
    } else {
      if (c.max_token_len <= 0) return GRPO_ERR_INVALID;
      for (int32_t i = 0; i < n_rows_in; ++i)
        if (row_len[i] > c.max_token_len) return GRPO_ERR_TOKEN_BUDGET;
      for (int32_t i = 0; i < n_steps; ++i) {
        dynamic_bins(c, i * mini, (i + 1) * mini, row_len, p);
        p.step_chunk_off.push_back((int32_t)p.chunk_row_off.size() - 1);
      }
    }
    p.row_pad.assign(p.row_src.size(), 0);
    p.row_gpu.assign(p.row_src.size(), 0);
    p.row_rollout = p.row_src;
  }

  const int32_t n_rows = (int32_t)p.row_src.size();
  const int32_t n_chunks = (int32_t)p.chunk_row_off.size() - 1;
  out->n_rows = n_rows;
  out->n_chunks = n_chunks;
  out->n_steps = n_steps;
  out->n_micro = p.n_micro;
  out->q = p.q;
  out->n_pad_rows = (int32_t)std::count(p.row_pad.begin(), p.row_pad.end(), 1);
  out->needs_old_logp_cache = (n_steps > 1 && !c.use_rollout_logprobs) ? 1 : 0;
  if (n_rows > out->cap_rows || n_chunks > out->cap_chunks || n_steps > out->cap_steps)
    return GRPO_ERR_CAPACITY;

  auto put = [](int32_t* dst, const std::vector<int32_t>& v) {
    if (dst && !v.empty()) std::memcpy(dst, v.data(), v.size() * sizeof(int32_t));
  };
  put(out->row_src, p.row_src);
  put(out->row_pad, p.row_pad);
  put(out->row_gpu, p.row_gpu);
  put(out->row_rollout, p.row_rollout);
  put(out->chunk_row_off, p.chunk_row_off);
  put(out->step_chunk_off, p.step_chunk_off);
  put(out->step_in_row_off, p.step_in_row_off);
  if (out->inv_perm) {
    for (int32_t i = 0; i < n_rows_in; ++i) out->inv_perm[i] = -1;
    for (int32_t j = 0; j < n_rows; ++j)
      if (!p.row_pad[j]) out->inv_perm[p.row_src[j]] = j;
  }
  for (int32_t ch = 0; ch < n_chunks; ++ch) {
    int64_t tok = 0;
    for (int32_t j = p.chunk_row_off[ch]; j < p.chunk_row_off[ch + 1]; ++j) tok += row_len[p.row_src[j]];
    if (out->chunk_tokens) out->chunk_tokens[ch] = tok;
  }
  for (int32_t s = 0; s < n_steps; ++s) {
    int64_t n_tok = 0;
    int32_t n_row = 0;
    const int32_t a = p.chunk_row_off[p.step_chunk_off[s]];
    const int32_t b = p.chunk_row_off[p.step_chunk_off[s + 1]];
    for (int32_t j = a; j < b; ++j) {
      if (p.row_pad[j]) continue;  // padding rows are masked: no valid token, no row
      const int32_t v = row_valid[p.row_src[j]];
      n_tok += v;
      n_row += v > 0;
    }
    if (out->step_valid_tokens) out->step_valid_tokens[s] = n_tok;
    if (out->step_valid_rows) out->step_valid_rows[s] = n_row;
  }
  return GRPO_OK;
}

extern "C" GRPO_API int grpo_plan_token_index(const grpo_plan* plan, int32_t n_rows_in,
                                              const int64_t* row_tok_off, int64_t* tok_src,
                                              int64_t cap, int64_t* n_out) {
  if (!plan || !row_tok_off || !n_out || n_rows_in < 0) return GRPO_ERR_INVALID;
  if (plan->n_rows > 0 && (!plan->row_src || !plan->row_pad)) return GRPO_ERR_INVALID;
  int64_t n = 0;
  for (int32_t j = 0; j < plan->n_rows; ++j) {
    const int32_t r = plan->row_src[j];
    if (r < 0 || r >= n_rows_in) return GRPO_ERR_INVALID;
    n += row_tok_off[r + 1] - row_tok_off[r];
  }
  *n_out = n;
  if (n > cap) return GRPO_ERR_CAPACITY;
  if (n > 0 && !tok_src) return GRPO_ERR_INVALID;
  int64_t t = 0;
  for (int32_t j = 0; j < plan->n_rows; ++j) {
    const int32_t r = plan->row_src[j];
    const bool pad = plan->row_pad[j] != 0;
    for (int64_t i = row_tok_off[r]; i < row_tok_off[r + 1]; ++i) tok_src[t++] = pad ? -1 - i : i;
  }
  return GRPO_OK;
}

extern "C" GRPO_API int grpo_plan_token_weights(const grpo_plan* plan, int32_t n_rows_in,
                                                const int64_t* row_tok_off, const int32_t* row_valid,
                                                int32_t agg, int64_t* step_divisor, float* w_tok,
                                                float* step_grad_scale) {
  if (!plan || !row_tok_off || !row_valid || !step_divisor || n_rows_in < 0 || plan->n_steps < 0)
    return GRPO_ERR_INVALID;
  if (agg != GRPO_AGG_TOKEN_MEAN && agg != GRPO_AGG_SEQ_MEAN_TOKEN_SUM && agg != GRPO_AGG_SEQ_MEAN_TOKEN_MEAN)
    return GRPO_ERR_INVALID;
  if (row_tok_off[0] != 0) return GRPO_ERR_INVALID;
  for (int32_t r = 0; r < n_rows_in; ++r) {
    const int64_t len = row_tok_off[r + 1] - row_tok_off[r];
    if (len < 0 || row_valid[r] < 0 || row_valid[r] > len) return GRPO_ERR_INVALID;
  }
  const int32_t* so = plan->step_in_row_off;
  if (!so || so[0] != 0 || so[plan->n_steps] != n_rows_in) return GRPO_ERR_INVALID;
  for (int32_t s = 0; s < plan->n_steps; ++s)
    if (so[s + 1] < so[s]) return GRPO_ERR_INVALID;
  for (int32_t s = 0; s < plan->n_steps; ++s) {
    int64_t N = 0, B = 0;
    for (int32_t r = so[s]; r < so[s + 1]; ++r) {
      N += row_valid[r];
      B += row_valid[r] >= 1;
    }
    step_divisor[s] = agg == GRPO_AGG_TOKEN_MEAN ? N : B;
    // the one division of the step, rounded once from float64 to float
    if (step_grad_scale) step_grad_scale[s] = (float)(1.0 / (double)(step_divisor[s] > 1 ? step_divisor[s] : 1));
    if (!w_tok) continue;
    for (int32_t r = so[s]; r < so[s + 1]; ++r) {
      const float w = agg == GRPO_AGG_SEQ_MEAN_TOKEN_MEAN
                          ? (float)(1.0 / (double)(row_valid[r] > 1 ? row_valid[r] : 1))
                          : 1.f;
      for (int64_t t = row_tok_off[r]; t < row_tok_off[r + 1]; ++t) w_tok[t] = w;
    }
  }
  return GRPO_OK;
}
