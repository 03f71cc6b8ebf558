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

// The same pair with the maximum kept in log2 units (m2 = max * log2(e)): the exponent of
// every element is then a single fma(x, log2e, -m2) and the shift cancels exactly in
// lse2 = m2 + log2(s), whatever the rounding of m2.
__device__ __forceinline__ MS ms2_combine(MS a, MS b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return {m, 0.f};
  return {m, a.s * ex2(a.m - m) + b.s * ex2(b.m - m)};
}

// Warp maximum of a float in one reduction instruction (NaN inputs are ignored, as fmaxf does).
__device__ __forceinline__ float warp_max_f32(float x) {
  float r;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}

// The warp's log2-domain (shift, sum) pairs combined: the largest shift M by one reduction,
// every lane's sum rescaled to it, the sums added by a fixed pairwise tree. Lane 0's result
// is the warp's (its order of additions is fixed). A warp without mass gives (-inf, 0).
__device__ __forceinline__ MS warp_ms2(MS v) {
  const float M = warp_max_f32(v.m);
  float s = M == -INFINITY ? 0.f : v.s * ex2(v.m - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return {M, s};
}

// The partials of each W-lane group of the warp (W a power of two, at most 32) combined by a
// fixed pairwise tree: lane g*W ends with group g's result, the same bits wherever the group
// sits in the warp.
template <int W>
__device__ __forceinline__ MS group_tree_ms2(MS v) {
  static_assert(W >= 1 && W <= 32 && (W & (W - 1)) == 0, "power of two");
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1)
    v = ms2_combine(v, MS{__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.s, o)});
  return v;
}

// Fold N more values into a log2-domain online pair (one rescale per call).
// Pairwise (tree) reductions of a register array: log2(N) dependent steps instead of N, so
// a thread's block of exponentials never waits on one long add chain. The order is fixed.
template <int N>
__device__ __forceinline__ float tree_max(const float (&x)[N]) {
  static_assert((N & (N - 1)) == 0, "power of two");
  float t[N];
#pragma unroll
  for (int i = 0; i < N; ++i) t[i] = x[i];
#pragma unroll
  for (int w = N / 2; w >= 1; w /= 2)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = fmaxf(t[i], t[i + w]);
  return t[0];
}

// Fixed-shape pairwise sum (t[i] += t[i + w], w = N/2, ..., 1), in place. PK: the levels with
// w >= 2 use packed two-lane adds (each lane adds the same two operands as the scalar tree, so
// the result is the same bits); PK = false keeps every add scalar (fewer register pairs).
template <int N, bool PK = true>
__device__ __forceinline__ float tree_sum(float (&t)[N]) {
  static_assert((N & (N - 1)) == 0, "power of two");
  if constexpr (PK) {
#pragma unroll
    for (int w = N / 2; w >= 2; w /= 2)
#pragma unroll
      for (int i = 0; i < w; i += 2) {
        const float2 r = __fadd2_rn(make_float2(t[i], t[i + 1]), make_float2(t[i + w], t[i + w + 1]));
        t[i] = r.x;
        t[i + 1] = r.y;
      }
    if (N >= 2) t[0] = t[0] + t[1];
  } else {
#pragma unroll
    for (int w = N / 2; w >= 1; w /= 2)
#pragma unroll
      for (int i = 0; i < w; ++i) t[i] = t[i] + t[i + w];
  }
  return t[0];
}

// 2^(x log2 e - sh) for a pair, the argument by one packed fused multiply-add per pair.
__device__ __forceinline__ float2 ex2_pair(float x0, float x1, float sh) {
  const float2 t = __ffma2_rn(make_float2(x0, x1), make_float2(kLog2e, kLog2e), make_float2(-sh, -sh));
  return make_float2(ex2(t.x), ex2(t.y));
}

// Fold N more values into a log2-domain online pair: one rescale per call, the N
// exponentials independent, summed by a fixed tree. Branch-free: while every value so far is
// -inf the shift is 0 and the sum stays 0.
template <int N>
__device__ __forceinline__ void online2(MS& acc, float (&x)[N]) {
  const float nm = fmaxf(acc.m, tree_max(x) * kLog2e);
  const bool none = nm == -INFINITY;
  const float scale = none ? 1.f : ex2(acc.m - nm);  // ex2(-inf) = 0 on the first finite block
  const float sh = none ? 0.f : nm;
#pragma unroll
  for (int i = 0; i < N; ++i) x[i] = ex2(fmaf(x[i], kLog2e, -sh));
  acc.s = fmaf(acc.s, scale, tree_sum(x));
  acc.m = nm;
}

// Lazy variant: exponentials are taken against the current shift, and the block's maximum
// is only computed when the block sum leaves the safe range (> 2^64, inf or NaN), which for
// real logits happens about once per thread and row (the first block, shift -inf). Exact in
// the same sense as online2: the sum carries its scale, and lse2 = m + log2(s) either way.
template <int N, bool PK = true>
__device__ __forceinline__ void lazy_online2(MS& acc, float (&x)[N]) {
  // the first block takes its first value as the shift (the sum is still 0, so any shift is
  // exact); a block rising more than 2^64 above it falls back to the max-based update
  if (acc.m == -INFINITY) acc.m = x[0] * kLog2e;
  float e[N];
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    if constexpr (PK) {
      const float2 p = ex2_pair(x[i], x[i + 1], acc.m);
      e[i] = p.x;
      e[i + 1] = p.y;
    } else {
      e[i] = ex2(fmaf(x[i], kLog2e, -acc.m));
      e[i + 1] = ex2(fmaf(x[i + 1], kLog2e, -acc.m));
    }
  }
  const float bs = tree_sum<N, PK>(e);
  if (bs <= 1.8446744e19f) {  // false for inf and NaN
    acc.s += bs;
    return;
  }
  online2<N>(acc, x);
}

// (max, sum e, sum e*x) triple for the entropy term: s2 / s = sum_v p_v z_v.
struct MS3 {
  float m, s, s2;
};

// natural-log units (max in logit units)
__device__ __forceinline__ MS3 ms3_combine(MS3 a, MS3 b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return {m, 0.f, 0.f};
  const float fa = ex2((a.m - m) * kLog2e), fb = ex2((b.m - m) * kLog2e);
  return {m, a.s * fa + b.s * fb, a.s2 * fa + b.s2 * fb};
}

// log2 units (max kept as max * log2(e))
__device__ __forceinline__ MS3 ms3_combine2(MS3 a, MS3 b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return {m, 0.f, 0.f};
  const float fa = ex2(a.m - m), fb = ex2(b.m - m);
  return {m, a.s * fa + b.s * fb, a.s2 * fa + b.s2 * fb};
}

template <bool LOG2>
__device__ __forceinline__ MS3 warp_ms3(MS3 v) {
  if constexpr (LOG2) {
    // as warp_ms2: one maximum, one rescale per lane, two fixed addition trees
    const float M = warp_max_f32(v.m);
    const float f = M == -INFINITY ? 0.f : ex2(v.m - M);
    float s = v.s * f, s2 = v.s2 * f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, o);
      s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    return {M, s, s2};
  } else {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      MS3 w{__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.s, o),
            __shfl_xor_sync(0xffffffffu, v.s2, o)};
      v = ms3_combine(v, w);
    }
    return v;
  }
}

template <int W>
__device__ __forceinline__ MS3 group_tree_ms3(MS3 v) {
  static_assert(W >= 1 && W <= 32 && (W & (W - 1)) == 0, "power of two");
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1)
    v = ms3_combine2(v, MS3{__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.s, o),
                            __shfl_xor_sync(0xffffffffu, v.s2, o)});
  return v;
}

// lazy_online2 that also accumulates sum e*x (log2-domain shift, natural-unit x). Pairs are
// combined as they are produced, so only half-width arrays of partial sums stay live.
template <int N>
__device__ __forceinline__ void e_pairs(const float (&x)[N], float sh, float (&pe)[N / 2], float (&px)[N / 2]) {
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const float e0 = ex2(fmaf(x[2 * i], kLog2e, -sh)), e1 = ex2(fmaf(x[2 * i + 1], kLog2e, -sh));
    pe[i] = e0 + e1;
    // p log p -> 0 as p -> 0: an element with no mass (a -inf logit) adds nothing to sum p z
    px[i] = (e0 != 0.f ? e0 * x[2 * i] : 0.f) + (e1 != 0.f ? e1 * x[2 * i + 1] : 0.f);
  }
}

// Block sums (sum e, sum e*x) of N values without the no-mass guard, in packed two-lane
// arithmetic: groups of four elements give lane j the elements 4g + j and 4g + 2 + j, the
// groups are summed by a fixed pairwise tree, and the two lanes are added last. e * x is NaN
// only where a logit is -inf (or the row is not finite at all), which the caller detects on
// the block sum.
template <int N>
__device__ __forceinline__ void e_sums_packed(const float (&x)[N], float sh, float& se, float& sx) {
  static_assert(N % 4 == 0 && (((N / 4) & (N / 4 - 1)) == 0), "N / 4 a power of two");
  float2 s[N / 4], p[N / 4];
#pragma unroll
  for (int g = 0; g < N / 4; ++g) {
    const float2 xa = make_float2(x[4 * g], x[4 * g + 1]), xb = make_float2(x[4 * g + 2], x[4 * g + 3]);
    const float2 ea = ex2_pair(xa.x, xa.y, sh), eb = ex2_pair(xb.x, xb.y, sh);
    s[g] = __fadd2_rn(ea, eb);
    p[g] = __ffma2_rn(eb, xb, __fmul2_rn(ea, xa));
  }
#pragma unroll
  for (int w = N / 8; w >= 1; w /= 2)
#pragma unroll
    for (int g = 0; g < w; ++g) {
      s[g] = __fadd2_rn(s[g], s[g + w]);
      p[g] = __fadd2_rn(p[g], p[g + w]);
    }
  se = s[0].x + s[0].y;
  sx = p[0].x + p[0].y;
}

// `guarded` is set when the block needed the no-mass guard (or the rescue path, which uses
// it): only then can the block hold a -inf logit.
template <int N>
__device__ __forceinline__ void lazy_online3(MS3& acc, const float (&x)[N], bool& guarded) {
  if (acc.m == -INFINITY) acc.m = x[0] * kLog2e;
  float pe[N / 2], px[N / 2];
  float bs, bx;
  e_sums_packed<N>(x, acc.m, bs, bx);
  if (bs <= 1.8446744e19f) {
    if (bx != bx) {  // a -inf logit in the block: redo it with no-mass elements adding nothing
      e_pairs<N>(x, acc.m, pe, px);
      bx = tree_sum(px);
      guarded = true;
    }
    acc.s += bs;
    acc.s2 += bx;
    return;
  }
  guarded = true;
  float gm = x[0];
#pragma unroll
  for (int i = 1; i < N; ++i) gm = fmaxf(gm, x[i]);
  const float nm = fmaxf(acc.m, gm * kLog2e);
  const bool none = nm == -INFINITY;
  const float scale = none ? 1.f : ex2(acc.m - nm);
  e_pairs<N>(x, none ? 0.f : nm, pe, px);
  acc.s = fmaf(acc.s, scale, tree_sum(pe));
  acc.s2 = fmaf(acc.s2, scale, tree_sum(px));
  acc.m = nm;
}

// Per-token scalar epilogue: log-prob, ratio, clipped surrogate, gradient coefficient.
struct TokenOut {
  float logp, loss, coef;
  bool clipped, nonfinite;
};

// Largest |LSE| (natural units) of a row whose results this library vouches for. The
// log-prob itself is formed without cancellation at any magnitude (the callers compute it as
// (z_y - shift) - log(sum) from their exact shift). Pass 2's exponent argument and the
// entropy's LSE - E_p[z], though, round at the scale of the LSE: within 4096 that is below
// 2.5e-4, beyond it the token is reported non-finite rather than returned degraded. Trained
// models' logits are in the tens.
constexpr float kLseMax = 4096.f;

// logp: the target's log-prob; in_range: |LSE| <= kLseMax (else the token reports NaN)
__device__ __forceinline__ TokenOut token_epilogue(float logp, bool in_range, bool has_old, float old,
                                                  float A, float eps, float scale) {
  TokenOut o;
  o.logp = in_range ? logp : __int_as_float(0x7fc00000);
  const float r = has_old ? expf(o.logp - old) : 1.f;
  const float lo = 1.f - eps, hi = 1.f + eps;
  const float rc = fminf(fmaxf(r, lo), hi);
  o.loss = -fminf(r * A, rc * A);
  o.clipped = (A > 0.f && r > hi) || (A < 0.f && r < lo);
  o.coef = o.clipped ? 0.f : A * r * scale;
  o.nonfinite = !isfinite(o.logp) || !isfinite(o.loss) || !isfinite(o.coef);
  return o;
}

// Regularisers sent through the same aggregation: kl_coef * k(logp, ref) with
// k1 = logp - ref or k3 = exp(ref - logp) - (ref - logp) - 1 (gradient folded into the
// (softmax - onehot) coefficient), and an entropy bonus -ent_coef * H (its loss part here; its
// gradient ent_coef * p (z - E_p z) is added by the vocabulary pass).
__device__ __forceinline__ void apply_terms(TokenOut& o, float scale, int kl_kind, float kl_coef, float ref,
                                            float ent_coef, float H) {
  if (kl_kind == GRPO_KL_K1 || kl_kind == GRPO_KL_K3) {
    const float d = ref - o.logp;
    float k, dk;
    if (kl_kind == GRPO_KL_K1) {
      k = -d;
      dk = 1.f;
    } else {
      const float ed = expf(d);
      k = ed - d - 1.f;
      dk = 1.f - ed;
    }
    o.loss += kl_coef * k;
    o.coef -= kl_coef * dk * scale;
  }
  if (ent_coef != 0.f) o.loss -= ent_coef * H;
  o.nonfinite = o.nonfinite || !isfinite(o.loss) || !isfinite(o.coef);
}

// ---- shared-memory, mbarrier, bulk-copy and cluster primitives (inline PTX, sm_90+) ----------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Acquire at cluster scope: pairs with a peer CTA's release-arrive on this barrier, so the
// peer's shared::cluster stores made before its arrive are visible after the wait.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Arrive on an mbarrier that lives in a peer CTA's shared memory (address from mapa),
// releasing this thread's earlier shared::cluster stores to that CTA.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Relaxed arrive (no fence) on an mbarrier in a peer CTA's shared memory: for a signal that
// publishes no data of this thread's.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Relaxed arrive that also raises the phase's expected transaction bytes (the data comes by
// st.async, whose completion the phase tracks; this thread publishes nothing).
__device__ __forceinline__ void mbar_arrive_expect_tx_relaxed(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Asynchronous stores into a peer CTA's shared memory (cluster addresses from mapa), each
// completing its bytes on an mbarrier of that CTA: the reader sees the data once the phase
// completes, and the writer waits for nothing.
__device__ __forceinline__ void st_async_v2f32(uint32_t cluster_addr, float x, float y, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
               ::"r"(cluster_addr), "f"(x), "f"(y), "r"(cluster_bar) : "memory");
}

__device__ __forceinline__ void st_async_f32(uint32_t cluster_addr, float x, uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];"
               ::"r"(cluster_addr), "f"(x), "r"(cluster_bar) : "memory");
}

__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase: gives up after ~1 s (or 2^24 polls), raises *abort and
// returns false. Once *abort is set no later wait blocks, so a broken pipeline still lets
// the kernel run to its end and report kFlagWaitTimeout instead of hanging.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (*abort) return false;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1; i < (1u << 24); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && global_timer_ns() - t0 > 1000000000ull) break;
    if (*abort) return false;
  }
  *abort = 1;
  return false;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort);
}

static __device__ __noinline__ bool mbar_wait_cluster_slow(uint64_t* bar, uint32_t parity,
                                                          volatile int* abort) {
  if (*abort) return false;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1; i < (1u << 24); ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 255u) == 0 && global_timer_ns() - t0 > 1000000000ull) break;
    if (*abort) return false;
  }
  *abort = 1;
  return false;
}

__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                          volatile int* abort) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  return mbar_wait_cluster_slow(bar, parity, abort);
}

// One contiguous global -> shared bulk copy completing on `bar` (16-byte aligned addresses,
// size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA in the cluster; release/acquire orders shared-memory writes
// before the barrier with reads from other CTAs after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ uint32_t mapa_u32(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace grpo

#define GRPO_CUDA_TRY(expr)                   \
  do {                                        \
    if ((expr) != cudaSuccess) {              \
      (void)cudaGetLastError();               \
      return GRPO_ERR_CUDA;                   \
    }                                         \
  } while (0)
