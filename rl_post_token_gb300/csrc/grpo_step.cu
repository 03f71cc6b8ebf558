// Step-level kernels: the group advantage with its token broadcast, and the step finish
// (float64 loss sum in a fixed order, metrics, skip on non-finite, deferred 1/max(N,1)).
//
// Sources: "03 Data Protocol and Batch Lifecycle" (uid groups; the scalar advantage broadcast
// to tokens and multiplied by the response mask); "How a context-compaction step fits a
// variable number of rows into one batch" (advantage once per rollout, copied to its rows,
// padding rows 0; one division by the step's valid tokens); "Sizing mini-batches and
// micro-batches" ("The hard part: deferred normalization": scale by 1/max(sum, 1), then clip,
// then step; "Metric roll-up": counts are summed, the loss is token-weighted; "The
// poisoned-window countdown": a non-finite chunk discards the accumulation window).
#include <algorithm>
#include <cstddef>

#include "grpo_common.cuh"

namespace grpo {

// One thread per group; float64 with explicit round-to-nearest operations (no fused
// multiply-add), so the float32 result is the correctly rounded value of the plain formula.
__global__ void adv_group_kernel(const float* __restrict__ rewards, int32_t n, int32_t G,
                                 double eps, int32_t unbiased, float* __restrict__ adv) {
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t g0 = g * G;
  if (g0 >= n) return;
  if (G < 2 && unbiased) {
    for (int32_t i = 0; i < G; ++i) adv[g0 + i] = 0.f;
    return;
  }
  double total = 0.0;
  for (int32_t i = 0; i < G; ++i) total = __dadd_rn(total, (double)rewards[g0 + i]);
  const double mean = __ddiv_rn(total, (double)G);
  double ss = 0.0;
  for (int32_t i = 0; i < G; ++i) {
    const double d = __dsub_rn((double)rewards[g0 + i], mean);
    ss = __dadd_rn(ss, __dmul_rn(d, d));
  }
  const double var = __ddiv_rn(ss, (double)(unbiased ? G - 1 : G));
  const double den = __dadd_rn(__dsqrt_rn(var), eps);
  for (int32_t i = 0; i < G; ++i)
    adv[g0 + i] = __double2float_rn(__ddiv_rn(__dsub_rn((double)rewards[g0 + i], mean), den));
}

__global__ void adv_broadcast_kernel(const float* __restrict__ adv,
                                     const int32_t* __restrict__ row_rollout,
                                     const int64_t* __restrict__ row_tok_off, int32_t n_rows,
                                     float* __restrict__ adv_tok) {
  for (int64_t r = blockIdx.x; r < n_rows; r += gridDim.x) {
    const int32_t ro = row_rollout ? row_rollout[r] : (int32_t)r;
    const float v = ro < 0 ? 0.f : adv[ro];
    const int64_t a = row_tok_off[r], b = row_tok_off[r + 1];
    for (int64_t t = a + threadIdx.x; t < b; t += blockDim.x) adv_tok[t] = v;
  }
}

constexpr int kFinishCtas = 8;       // one cluster
constexpr int kFinishThreads = 256;  // per CTA

// One term of the step sum: the token's loss, times its aggregation weight when there is one
// (the product of two floats is exact in float64).
template <bool W>
__device__ __forceinline__ double weighted(const float* __restrict__ loss_tok, const float* __restrict__ w_tok,
                                           int64_t i) {
  return W ? (double)w_tok[i] * (double)loss_tok[i] : (double)loss_tok[i];
}

__device__ __forceinline__ double ld_dsmem_f64(uint32_t addr) {
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(addr) : "memory");
  return v;
}

// One cluster of kFinishCtas CTAs: CTA r sums the r-th contiguous eighth of the step's
// (weighted) per-token losses in float64 (thread-strided partial sums, then a fixed tree);
// CTA 0 adds the eight partials in rank order through distributed shared memory. The order
// depends only on n. Then the metrics, the status, the divisor, and the counter reset.
template <bool W>
__global__ void __launch_bounds__(kFinishThreads)
finish_kernel(grpo_step_acc* acc, const float* __restrict__ loss_tok, const float* __restrict__ w_tok,
              int64_t n, int64_t expected_N, int64_t divisor) {
  __shared__ double sh[kFinishThreads];
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_ctarank();
  const int64_t lo = n * (int64_t)rank / kFinishCtas, hi = n * (int64_t)(rank + 1) / kFinishCtas;
  double s = 0.0;
  int64_t i = lo + tid;
  for (; i + 3 * kFinishThreads < hi; i += 4 * kFinishThreads) {
    const double a0 = weighted<W>(loss_tok, w_tok, i), a1 = weighted<W>(loss_tok, w_tok, i + kFinishThreads);
    const double a2 = weighted<W>(loss_tok, w_tok, i + 2 * kFinishThreads);
    const double a3 = weighted<W>(loss_tok, w_tok, i + 3 * kFinishThreads);
    s += a0;
    s += a1;
    s += a2;
    s += a3;
  }
  for (; i < hi; i += kFinishThreads) s += weighted<W>(loss_tok, w_tok, i);
  sh[tid] = s;
  __syncthreads();
  for (int w = kFinishThreads / 2; w > 0; w >>= 1) {
    if (tid < w) sh[tid] += sh[tid + w];
    __syncthreads();
  }
  cluster_sync_all();  // every CTA's partial is in its sh[0]
  if (rank == 0 && tid == 0) {
    double total = 0.0;
    const uint32_t a0 = smem_u32(&sh[0]);
    for (int r = 0; r < kFinishCtas; ++r) total += ld_dsmem_f64(mapa_u32(a0, (uint32_t)r));
    grpo_step_result res;
    res.loss_sum = total;
    res.n_valid = (int64_t)acc->n_valid;
    res.n_clipped = (int64_t)acc->n_clipped;
    res.n_nonfinite = (int64_t)acc->n_nonfinite;
    res.n_tokens = (int64_t)acc->n_tokens;
    res.kernel_flags = (int32_t)acc->flags;
    const double N = (double)(res.n_valid > 1 ? res.n_valid : 1);
    const int64_t D = divisor >= 0 ? divisor : res.n_valid;
    res.loss = res.loss_sum / (double)(D > 1 ? D : 1);
    res.clipfrac = (double)res.n_clipped / N;
    acc->divisor = D;
    if (res.kernel_flags)
      res.status = GRPO_ERR_KERNEL;
    else if (expected_N >= 0 && expected_N != res.n_valid)
      res.status = GRPO_ERR_N_MISMATCH;
    else if (res.n_nonfinite > 0)
      res.status = GRPO_STEP_SKIPPED_NONFINITE;
    else
      res.status = GRPO_OK;
    acc->result = res;
    acc->n_valid = acc->n_clipped = acc->n_nonfinite = acc->n_tokens = 0;
    acc->flags = 0;
  }
  cluster_sync_all();  // no CTA leaves while CTA 0 may still read its partial
}

template <bool W>
int launch_finish(grpo_step_acc* acc, const float* loss_tok, const float* w_tok, int64_t n, int64_t expected_N,
                  int64_t divisor, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kFinishCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(kFinishCtas, 1, 1);
  cfg.blockDim = dim3(kFinishThreads, 1, 1);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  GRPO_CUDA_TRY(cudaLaunchKernelEx(&cfg, finish_kernel<W>, acc, loss_tok, w_tok, n, expected_N, divisor));
  return GRPO_OK;
}

// Registered gradient buffer: zeroed when the step is discarded, else (deferred mode) scaled
// once by 1/max(D, 1), D the step's divisor; a kept step in non-deferred mode leaves it untouched.
template <typename T>
__global__ void grad_finish_kernel(T* __restrict__ g, int64_t n, const grpo_step_acc* acc,
                                   int32_t deferred) {
  const int32_t status = acc->result.status;
  const bool discard = status != GRPO_OK;
  if (!discard && !deferred) return;
  const int64_t D = acc->divisor;
  const float f = discard ? 0.f : (float)(1.0 / (double)(D > 1 ? D : 1));
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float v = discard ? 0.f : (float)g[i] * f;
    g[i] = (T)v;
  }
}

// One bounded wait that nothing completes: the barrier's first phase never ends, so the wait
// gives up at its limit and the kernel raises the wait-timeout flag, as a pipelined kernel
// whose producer or peer stopped would.
__global__ void wait_timeout_selftest_kernel(grpo_step_acc* acc) {
  __shared__ uint64_t bar;
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    s_abort = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0u, &s_abort)) atomicOr(&acc->flags, kFlagWaitTimeout);
}

}  // namespace grpo

using namespace grpo;

extern "C" GRPO_API int grpo_selftest_wait_timeout(grpo_step_acc* acc, void* stream) {
  if (!acc) return GRPO_ERR_INVALID;
  wait_timeout_selftest_kernel<<<1, 32, 0, as_stream(stream)>>>(acc);
  GRPO_CUDA_TRY(cudaGetLastError());
  return GRPO_OK;
}

extern "C" GRPO_API int grpo_group_advantage(const float* rewards, int32_t n_rollouts,
                                             int32_t group_size, float eps,
                                             int32_t unbiased_std, float* adv_out,
                                             const int32_t* row_rollout,
                                             const int64_t* row_tok_off, int32_t n_rows,
                                             float* adv_tok, void* stream) {
  if (n_rollouts < 0 || group_size <= 0 || n_rollouts % group_size != 0) return GRPO_ERR_INVALID;
  if (n_rollouts > 0 && (!rewards || !adv_out)) return GRPO_ERR_INVALID;
  if (adv_tok && (!row_tok_off || n_rows < 0)) return GRPO_ERR_INVALID;
  if (adv_tok && !row_rollout && n_rows != n_rollouts) return GRPO_ERR_INVALID;
  const cudaStream_t st = as_stream(stream);
  const int32_t n_groups = n_rollouts / group_size;
  if (n_groups > 0) {
    const int thr = 128;
    adv_group_kernel<<<(n_groups + thr - 1) / thr, thr, 0, st>>>(rewards, n_rollouts, group_size,
                                                                 (double)eps, unbiased_std, adv_out);
    GRPO_CUDA_TRY(cudaGetLastError());
  }
  if (adv_tok && n_rows > 0) {
    const int grid = std::min<int>(n_rows, sm_count() * 8);
    adv_broadcast_kernel<<<grid, 256, 0, st>>>(adv_out, row_rollout, row_tok_off, n_rows, adv_tok);
    GRPO_CUDA_TRY(cudaGetLastError());
  }
  return GRPO_OK;
}

extern "C" GRPO_API int grpo_finish_step_ex(grpo_step_acc* acc, const float* loss_tok, int64_t n_tok,
                                            const float* w_tok, int64_t divisor, int64_t expected_N,
                                            int32_t deferred, void* const* grad_bufs,
                                            const int64_t* grad_numels, const int32_t* grad_dtypes,
                                            int32_t n_bufs, grpo_step_result* result_host, void* stream) {
  if (!acc || n_tok < 0 || n_bufs < 0) return GRPO_ERR_INVALID;
  if (n_tok > 0 && !loss_tok) return GRPO_ERR_INVALID;
  if (n_bufs > 0 && (!grad_bufs || !grad_numels || !grad_dtypes)) return GRPO_ERR_INVALID;
  for (int32_t b = 0; b < n_bufs; ++b) {
    if (grad_dtypes[b] != GRPO_DTYPE_F32 && grad_dtypes[b] != GRPO_DTYPE_BF16) return GRPO_ERR_UNSUPPORTED;
    if (grad_numels[b] < 0 || (grad_numels[b] > 0 && !grad_bufs[b])) return GRPO_ERR_INVALID;
  }
  const cudaStream_t st = as_stream(stream);
  {
    const int rc = w_tok && n_tok > 0 ? launch_finish<true>(acc, loss_tok, w_tok, n_tok, expected_N, divisor, st)
                                      : launch_finish<false>(acc, loss_tok, nullptr, n_tok, expected_N, divisor, st);
    if (rc != GRPO_OK) return rc;
  }
  for (int32_t b = 0; b < n_bufs; ++b) {
    const int64_t n = grad_numels[b];
    if (n == 0) continue;
    const int grid = (int)std::min<int64_t>((n + 255) / 256, (int64_t)sm_count() * 8);
    if (grad_dtypes[b] == GRPO_DTYPE_F32)
      grad_finish_kernel<float><<<grid, 256, 0, st>>>(static_cast<float*>(grad_bufs[b]), n, acc, deferred);
    else
      grad_finish_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<__nv_bfloat16*>(grad_bufs[b]), n, acc,
                                                              deferred);
    GRPO_CUDA_TRY(cudaGetLastError());
  }
  if (!result_host) return GRPO_OK;
  GRPO_CUDA_TRY(cudaMemcpyAsync(result_host, &acc->result, sizeof(grpo_step_result),
                                cudaMemcpyDeviceToHost, st));
  GRPO_CUDA_TRY(cudaStreamSynchronize(st));
  return result_host->status;
}

extern "C" GRPO_API int grpo_finish_step(grpo_step_acc* acc, const float* loss_tok, int64_t n_tok,
                                         int64_t expected_N, int32_t deferred,
                                         void* const* grad_bufs, const int64_t* grad_numels,
                                         const int32_t* grad_dtypes, int32_t n_bufs,
                                         grpo_step_result* result_host, void* stream) {
  return grpo_finish_step_ex(acc, loss_tok, n_tok, nullptr, -1, expected_N, deferred, grad_bufs, grad_numels,
                             grad_dtypes, n_bufs, result_host, stream);
}

extern "C" GRPO_API const char* grpo_status_string(int status) {
  switch (status) {
    case GRPO_OK: return "ok";
    case GRPO_STEP_SKIPPED_NONFINITE: return "step skipped: non-finite log-prob or loss";
    case GRPO_ERR_INVALID: return "invalid argument";
    case GRPO_ERR_DIVISIBILITY: return "batch, mini and micro must divide exactly";
    case GRPO_ERR_ROLLOUT_COUNT: return "the step must hold exactly `batch` rollouts";
    case GRPO_ERR_TOKEN_BUDGET: return "a row is longer than max_token_len";
    case GRPO_ERR_INCOMPATIBLE: return "incompatible planner options";
    case GRPO_ERR_CAPACITY: return "output arrays too small";
    case GRPO_ERR_CUDA: return "CUDA runtime error";
    case GRPO_ERR_N_MISMATCH: return "counted N differs from the planned N";
    case GRPO_ERR_KERNEL: return "a bounded wait inside a kernel gave up";
    case GRPO_ERR_UNSUPPORTED: return "unsupported dtype or device";
    default: return "unknown status";
  }
}

extern "C" GRPO_API int grpo_version(void) { return 200; }

static_assert(sizeof(grpo_step_result) == 64, "grpo_step_result is 64 bytes");
static_assert(sizeof(grpo_step_acc) == 128, "grpo_step_acc is 128 bytes");
static_assert(offsetof(grpo_step_acc, result) == 64, "result sits in the second half");
static_assert(offsetof(grpo_step_acc, divisor) == 40, "divisor follows the flags");
