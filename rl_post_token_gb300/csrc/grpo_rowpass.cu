// Per-token-row vocabulary pass: log-softmax over V, gather of the sampled token's log-prob,
// ratio against pi_old, clipped surrogate, masking, and dlogits = coef * (softmax - onehot),
// without ever materialising the [T, V] float32 softmax.
//
// Sources ("Sizing mini-batches and micro-batches"): "The problem" (the log-softmax over the
// vocabulary of every completion token is the memory and time sink), "The hard part: deferred
// normalization" (token mean over the step, divide once by N), "pi_old must be frozen across
// the window" (ratio against the frozen pi_old, epsilon clip). The surrogate's formula is the
// standard PPO clip; the pages do not print it.
//
// Two kernels serve one entry point:
//  * row_l2_kernel      -- any dtype / V / alignment. A CTA owns a row: pass 1 streams the row
//                          from HBM with 16-byte loads keeping an online (max, sum-exp);
//                          pass 2 re-reads it (from L2 when the working set fits) and writes
//                          dlogits with 16-byte streaming stores.
//  * row_cluster_kernel -- bf16 rows with V % 8 == 0 and 16-byte aligned rows: a cluster of
//                          C CTAs splits each row; every CTA bulk-copies its slice into shared
//                          memory once (cp.async.bulk + mbarrier), both passes run from shared
//                          memory, and the CTAs exchange their (max, sum-exp) pairs and the
//                          target logit through distributed shared memory. HBM traffic is one
//                          read and one write of the row.
// Each row's reduction order depends only on V and the kernel's fixed shape, never on T or on
// how the step was chunked, so chunked and un-chunked calls agree bit for bit.
#include <cooperative_groups.h>

#include <algorithm>

#include "grpo_common.cuh"

namespace cg = cooperative_groups;

namespace grpo {

struct RowArgs {
  const void* logits;
  int64_t T, V, ld;
  const int64_t* tok_src;
  const int32_t* target;
  const float* old_logp;
  const float* adv;
  const uint8_t* mask;
  float eps, scale;
  void* dlogits;
  int64_t ld_out;
  float* loss_tok;
  float* logp_tok;
  grpo_step_acc* acc;
};

template <typename T>
struct Vec;

template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void unpack(const uint4& u, float (&f)[N]) {
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[N]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
  }
  __device__ __forceinline__ static float load1(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
  }
  __device__ __forceinline__ static void store1(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
  }
};

template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4& u, float (&f)[N]) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  __device__ __forceinline__ static uint4 pack(const float (&f)[N]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
  __device__ __forceinline__ static float load1(const float* p) { return *p; }
  __device__ __forceinline__ static void store1(float* p, float v) { *p = v; }
};

// Side inputs of one token row, resolved through tok_src.
struct TokMeta {
  int64_t idx;   // index into the per-token side arrays (-1 for padding rows)
  bool valid;    // mask = 1 and not a padding row
};

__device__ __forceinline__ TokMeta tok_meta(const RowArgs& a, int64_t row) {
  const int64_t src = a.tok_src ? a.tok_src[row] : row;
  TokMeta t;
  t.idx = src < 0 ? -1 : src;
  t.valid = src >= 0 && a.mask[src] != 0;
  return t;
}

// Counters a CTA accumulates and flushes once (integer: order-independent).
struct Counts {
  unsigned long long valid = 0, clipped = 0, nonfinite = 0, tokens = 0;
  __device__ void flush(grpo_step_acc* acc) {
    if (tokens) atomicAdd(reinterpret_cast<unsigned long long*>(&acc->n_tokens), tokens);
    if (valid) atomicAdd(reinterpret_cast<unsigned long long*>(&acc->n_valid), valid);
    if (clipped) atomicAdd(reinterpret_cast<unsigned long long*>(&acc->n_clipped), clipped);
    if (nonfinite) atomicAdd(reinterpret_cast<unsigned long long*>(&acc->n_nonfinite), nonfinite);
  }
};

// ------------------------------------------------------------------------------------------
// Generic kernel: one CTA per row at a time, persistent over rows.
// ------------------------------------------------------------------------------------------
template <typename T, int NT, int U, bool VEC>
__global__ void __launch_bounds__(NT) row_l2_kernel(RowArgs a) {
  constexpr int VN = Vec<T>::N;
  constexpr int NW = NT / 32;
  __shared__ float sh_m[NW], sh_s[NW];
  __shared__ float sh_lse, sh_coef;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t V = a.V;
  const int64_t nvec = VEC ? V / VN : 0;
  const int64_t tail0 = nvec * VN;
  Counts cnt;

  for (int64_t row = blockIdx.x; row < a.T; row += gridDim.x) {
    const TokMeta tm = tok_meta(a, row);
    const T* z = static_cast<const T*>(a.logits) + row * a.ld;
    T* dz = a.dlogits ? static_cast<T*>(a.dlogits) + row * a.ld_out : nullptr;
    if (!tm.valid) {
      // masked or padding row: nothing is read; loss, log-prob and dlogits are 0
      if (dz) {
        const uint4 zero = make_uint4(0, 0, 0, 0);
        for (int64_t j = tid; j < nvec; j += NT) __stcs(reinterpret_cast<uint4*>(dz) + j, zero);
        for (int64_t e = tail0 + tid; e < V; e += NT) Vec<T>::store1(dz + e, 0.f);
      }
      if (tid == 0) {
        cnt.tokens++;
        if (tm.idx >= 0) {
          a.loss_tok[tm.idx] = 0.f;
          if (a.logp_tok) a.logp_tok[tm.idx] = 0.f;
        }
      }
      continue;
    }
    const int32_t y = a.target[tm.idx];
    const bool ybad = y < 0 || (int64_t)y >= V;
    float zy = 0.f;
    if (tid == 0 && !ybad) zy = Vec<T>::load1(z + y);

    // pass 1: online max / sum of exp over the row
    MS acc{-INFINITY, 0.f};
    const uint4* zv = reinterpret_cast<const uint4*>(z);
    for (int64_t j0 = tid; j0 < nvec; j0 += (int64_t)NT * U) {
      float x[U][VN];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t j = j0 + (int64_t)u * NT;
        if (j < nvec) {
          Vec<T>::unpack(__ldg(zv + j), x[u]);
        } else {
#pragma unroll
          for (int i = 0; i < VN; ++i) x[u][i] = -INFINITY;
        }
      }
      float gm = x[0][0];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < VN; ++i) gm = fmaxf(gm, x[u][i]);
      if (gm > acc.m) {
        acc.s *= ex2((acc.m - gm) * kLog2e);
        acc.m = gm;
      }
      if (acc.m != -INFINITY) {
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int i = 0; i < VN; ++i) acc.s += ex2((x[u][i] - acc.m) * kLog2e);
      }
    }
    for (int64_t e = tail0 + tid; e < V; e += NT) {
      const float x = Vec<T>::load1(z + e);
      acc = ms_combine(acc, MS{x, 1.f});
    }

    // CTA reduction (fixed tree) and the per-token epilogue on thread 0
    MS w = warp_ms(acc);
    if (lane == 0) { sh_m[warp] = w.m; sh_s[warp] = w.s; }
    __syncthreads();
    if (warp == 0) {
      MS v = lane < NW ? MS{sh_m[lane], sh_s[lane]} : MS{-INFINITY, 0.f};
      v = warp_ms(v);
      if (lane == 0) {
        const float lse = v.m + logf(v.s);
        const TokenOut o = token_epilogue(ybad ? __int_as_float(0x7fc00000) : zy, lse, a.old_logp,
                                          tm.idx, a.adv[tm.idx], a.eps, a.scale);
        a.loss_tok[tm.idx] = o.loss;
        if (a.logp_tok) a.logp_tok[tm.idx] = o.logp;
        cnt.tokens++;
        cnt.valid++;
        cnt.clipped += o.clipped;
        cnt.nonfinite += o.nonfinite;
        sh_lse = lse;
        sh_coef = o.coef;
      }
    }
    __syncthreads();
    const float lse = sh_lse, coef = sh_coef;

    // pass 2: dlogits = coef * (softmax - onehot)
    if (dz) {
      uint4* dv = reinterpret_cast<uint4*>(dz);
      if (coef == 0.f) {
        const uint4 zero = make_uint4(0, 0, 0, 0);
        for (int64_t j = tid; j < nvec; j += NT) __stcs(dv + j, zero);
        for (int64_t e = tail0 + tid; e < V; e += NT) Vec<T>::store1(dz + e, 0.f);
      } else {
        for (int64_t j = tid; j < nvec; j += NT) {
          float x[VN];
          Vec<T>::unpack(__ldcs(zv + j), x);
#pragma unroll
          for (int i = 0; i < VN; ++i) x[i] = coef * ex2((x[i] - lse) * kLog2e);
          const int64_t off = (int64_t)y - j * VN;
          if (off >= 0 && off < VN) {
#pragma unroll
            for (int i = 0; i < VN; ++i)
              if (i == off) x[i] -= coef;
          }
          __stcs(dv + j, Vec<T>::pack(x));
        }
        for (int64_t e = tail0 + tid; e < V; e += NT) {
          float p = coef * ex2((Vec<T>::load1(z + e) - lse) * kLog2e);
          if (e == y) p -= coef;
          Vec<T>::store1(dz + e, p);
        }
      }
    }
    __syncthreads();  // sh_* are rewritten by the next row
  }
  if (tid == 0) cnt.flush(a.acc);
}

template <typename T, int NT, int U>
int launch_l2(const RowArgs& a, bool vec, int blocks_per_sm, cudaStream_t st) {
  const int64_t grid = std::min<int64_t>(a.T, (int64_t)sm_count() * blocks_per_sm);
  if (vec)
    row_l2_kernel<T, NT, U, true><<<(unsigned)grid, NT, 0, st>>>(a);
  else
    row_l2_kernel<T, NT, U, false><<<(unsigned)grid, NT, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? GRPO_OK : GRPO_ERR_CUDA;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

}  // namespace grpo

using namespace grpo;

extern "C" GRPO_API int grpo_logprob_loss_fwd_bwd(const void* logits, int32_t dtype, int64_t T,
                                                  int64_t V, int64_t ld, const int64_t* tok_src,
                                                  const int32_t* target, const float* old_logp,
                                                  const float* adv_tok, const uint8_t* mask,
                                                  float clip_eps, float grad_scale,
                                                  void* dlogits, int64_t ld_out, float* loss_tok,
                                                  float* logp_tok, grpo_step_acc* acc,
                                                  void* stream) {
  if (dtype != GRPO_DTYPE_F32 && dtype != GRPO_DTYPE_BF16) return GRPO_ERR_UNSUPPORTED;
  if (T < 0 || V < 1 || ld < V || !acc) return GRPO_ERR_INVALID;
  if (dlogits && ld_out < V) return GRPO_ERR_INVALID;
  if (T == 0) return GRPO_OK;
  if (!logits || !target || !adv_tok || !mask || !loss_tok) return GRPO_ERR_INVALID;
  if (V > (int64_t)INT32_MAX) return GRPO_ERR_INVALID;

  RowArgs a{logits, T, V, ld, tok_src, target, old_logp, adv_tok, mask, clip_eps, grad_scale,
            dlogits, ld_out, loss_tok, logp_tok, acc};
  const cudaStream_t st = as_stream(stream);
  const size_t es = dtype == GRPO_DTYPE_F32 ? 4 : 2;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool vec = al16(logits) && (ld * es) % 16 == 0 &&
                   (!dlogits || (al16(dlogits) && (ld_out * es) % 16 == 0));
  if (dtype == GRPO_DTYPE_BF16) {
    if (V >= 8192) return launch_l2<__nv_bfloat16, 1024, 2>(a, vec, 1, st);
    return launch_l2<__nv_bfloat16, 128, 2>(a, vec, 16, st);
  }
  if (V >= 8192) return launch_l2<float, 1024, 2>(a, vec, 1, st);
  return launch_l2<float, 128, 2>(a, vec, 16, st);
}
