// Internal helpers shared by the library's CUDA translation units (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "grpo.h"

namespace grpo {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)
constexpr float kLn2 = 0.6931471805599453f;    // ln(2)

// Bits of grpo_step_acc::flags raised by kernels (reported as result.kernel_flags).
constexpr unsigned kFlagWaitTimeout = 1u;   // a bounded mbarrier wait gave up
constexpr unsigned kFlagBadLaunch = 2u;     // a kernel saw a launch shape it cannot serve

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Multiprocessor count of the current device, cached per device ordinal.
int sm_count();

// One MUFU ex2 (PTX ex2.approx.ftz.f32: 2^x, relative error within 2^-22 per the PTX ISA).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round two floats to bf16 (nearest even) and pack them, lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Online (max, sum of exp(x - max)) pair, natural-log units.
struct MS {
  float m, s;
};

__device__ __forceinline__ MS ms_combine(MS a, MS b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return {m, 0.f};
  return {m, a.s * ex2((a.m - m) * kLog2e) + b.s * ex2((b.m - m) * kLog2e)};
}

__device__ __forceinline__ MS warp_ms(MS v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MS w{__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.s, o)};
    v = ms_combine(v, w);
  }
  return v;
}

// Per-token scalar epilogue: log-prob, ratio, clipped surrogate, gradient coefficient.
struct TokenOut {
  float logp, loss, coef;
  bool clipped, nonfinite;
};

__device__ __forceinline__ TokenOut token_epilogue(float zy, float lse, const float* old_logp,
                                                  int64_t idx, float A, float eps, float scale) {
  TokenOut o;
  o.logp = zy - lse;
  const float r = old_logp ? expf(o.logp - old_logp[idx]) : 1.f;
  const float lo = 1.f - eps, hi = 1.f + eps;
  const float rc = fminf(fmaxf(r, lo), hi);
  o.loss = -fminf(r * A, rc * A);
  o.clipped = (A > 0.f && r > hi) || (A < 0.f && r < lo);
  o.coef = o.clipped ? 0.f : A * r * scale;
  o.nonfinite = !isfinite(o.logp) || !isfinite(o.loss) || !isfinite(o.coef);
  return o;
}

}  // namespace grpo

#define GRPO_CUDA_TRY(expr)                   \
  do {                                        \
    if ((expr) != cudaSuccess) {              \
      (void)cudaGetLastError();               \
      return GRPO_ERR_CUDA;                   \
    }                                         \
  } while (0)
