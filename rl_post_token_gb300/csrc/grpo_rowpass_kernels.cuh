#pragma once
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
// Three kernels serve one entry point:
//  * row_l2_kernel      -- any dtype / V / alignment. A CTA owns a row: pass 1 streams the row
//                          from HBM with 16-byte loads keeping an online (max, sum-exp);
//                          pass 2 re-reads it (from L2 when the working set fits) and writes
//                          dlogits with 16-byte streaming stores.
//  * row_cluster_kernel -- bf16 (V % 8 == 0) or float32 (V % 4 == 0) rows, 16-byte aligned: a
//                          cluster of C CTAs splits each row; every CTA streams its slice
//                          through a shared-memory ring (cp.async.bulk + mbarrier), both passes
//                          run from shared memory, and the CTAs exchange their (shift, sum-exp)
//                          pairs and the target logit through distributed shared memory. HBM
//                          traffic is one read and one write of the row.
//  * row_fwd_kernel     -- the same split for forward-only calls without extra terms (the
//                          pi_old ahead pass): no per-row barrier, partials sent to CTA 0 and
//                          combined there by a dedicated warp, the same bits.
// Each row's reduction order depends only on V and the kernel's fixed shape, never on T or on
// how the step was chunked, so chunked and un-chunked calls agree bit for bit. The log-prob is
// formed as (z_y - shift) - log(sum) from the shift every term used, without cancellation;
// rows with |LSE| above kLseMax are reported non-finite.
#include <algorithm>
#include <type_traits>

#include "grpo_common.cuh"

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
  // regularisers (kl_kind 0 and ent_coef 0: none)
  int32_t kl_kind;
  float kl_coef;
  const float* ref_logp;
  float ent_coef;
  float* entropy_tok;
  const float* w_tok;  // per-token weight multiplying `scale` (an aggregation mode), or NULL
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

// Side inputs of one token row, resolved through tok_src. The instances with extra terms
// keep the token index in 32 bits (a call has fewer than 2^31 rows): the register it saves
// is what lets them run full-size chunks without spilling. The plain instances keep 64 bits,
// the layout their register allocation was tuned with.
template <int TERMS>
struct RowMeta {
  std::conditional_t<TERMS == 0, int64_t, int32_t> idx;  // index into the per-token side arrays (-1: padding)
  bool valid;    // mask = 1 and not a padding row
  int32_t y;     // target token id
  float A, old;  // advantage, pi_old log-prob
  float ref;     // reference-policy log-prob (KL term)
  float w;       // per-token weight of the gradient scale (aggregation mode)
};

__device__ __forceinline__ int64_t row_src(const RowArgs& a, int64_t row) {
  return a.tok_src ? a.tok_src[row] : row;
}

// TERMS is a set of kTerms* bits: the KL / entropy regularisers, the per-token weights.
constexpr int kTermsReg = 1;
constexpr int kTermsWeight = 2;

template <int TERMS>
__device__ __forceinline__ RowMeta<TERMS> row_meta(const RowArgs& a, int64_t src) {
  RowMeta<TERMS> m{src < 0 ? -1 : (decltype(RowMeta<TERMS>::idx))src, false, 0, 0.f, 0.f, 0.f, 1.f};
  if (src >= 0) {
    m.valid = a.mask[src] != 0;
    m.y = a.target[src];
    m.A = a.adv[src];
    m.old = a.old_logp ? a.old_logp[src] : 0.f;
    if (TERMS & kTermsReg) m.ref = a.ref_logp ? a.ref_logp[src] : 0.f;
    if (TERMS & kTermsWeight) m.w = a.w_tok[src];
  }
  return m;
}

// Row metadata fetched ahead of use: the token index two rows ahead and the side inputs one
// row ahead are in flight while the current row is processed, so the dependent global-load
// chain (index -> mask/target/advantage/pi_old) never sits on a row's critical path.
template <int TERMS>
struct MetaPipe {
  const RowArgs& a;
  int64_t stride;
  RowMeta<TERMS> next;
  int64_t src2;
  __device__ MetaPipe(const RowArgs& args, int64_t first, int64_t step) : a(args), stride(step) {
    next = first < a.T ? row_meta<TERMS>(a, row_src(a, first)) : RowMeta<TERMS>{-1, false, 0, 0.f, 0.f, 0.f, 1.f};
    src2 = first + step < a.T ? row_src(a, first + step) : -1;
  }
  // metadata of `row`; starts the loads for the rows after it
  __device__ RowMeta<TERMS> advance(int64_t row) {
    const RowMeta<TERMS> m = next;
    if (row + stride < a.T) next = row_meta<TERMS>(a, src2);
    src2 = row + 2 * stride < a.T ? row_src(a, row + 2 * stride) : -1;
    return m;
  }
};

// One dlogit with the entropy term, p (ea + eb z); an element with no mass stays 0.
__device__ __forceinline__ float ent_dz(float p, float z, float ea, float eb) {
  return p != 0.f ? p * fmaf(eb, z, ea) : 0.f;
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
template <typename T, int NT, int U, bool VEC, bool ENT, int TERMS>
__global__ void __launch_bounds__(NT) row_l2_kernel(RowArgs a) {
  constexpr int VN = Vec<T>::N;
  constexpr int NW = NT / 32;
  __shared__ float sh_m[NW], sh_s[NW], sh_s2[NW];
  __shared__ float sh_lse, sh_coef, sh_ez;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t V = a.V;
  const int64_t nvec = VEC ? V / VN : 0;
  const int64_t tail0 = nvec * VN;
  Counts cnt;

  MetaPipe<TERMS> pipe(a, blockIdx.x, gridDim.x);
  for (int64_t row = blockIdx.x; row < a.T; row += gridDim.x) {
    const auto tm = pipe.advance(row);
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
          if ((TERMS & kTermsReg) && a.entropy_tok) a.entropy_tok[tm.idx] = 0.f;
        }
      }
      continue;
    }
    const int32_t y = tm.y;
    const bool ybad = y < 0 || (int64_t)y >= V;
    float zy = 0.f;
    if (tid == 0 && !ybad) zy = Vec<T>::load1(z + y);

    // pass 1: online max / sum of exp over the row (and sum of exp * z for the entropy)
    MS acc{-INFINITY, 0.f};
    float acc_s2 = 0.f;
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
        const float f = ex2((acc.m - gm) * kLog2e);
        acc.s *= f;
        if (ENT) acc_s2 *= f;
        acc.m = gm;
      }
      if (acc.m != -INFINITY) {
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int i = 0; i < VN; ++i) {
            const float e = ex2((x[u][i] - acc.m) * kLog2e);
            acc.s += e;
            if (ENT && e != 0.f) acc_s2 = fmaf(e, x[u][i], acc_s2);  // no-mass elements add nothing
          }
      }
    }
    for (int64_t e = tail0 + tid; e < V; e += NT) {
      const float x = Vec<T>::load1(z + e);
      if (ENT) {
        const MS3 r = ms3_combine(MS3{acc.m, acc.s, acc_s2}, MS3{x, 1.f, x == -INFINITY ? 0.f : x});
        acc = MS{r.m, r.s};
        acc_s2 = r.s2;
      } else {
        acc = ms_combine(acc, MS{x, 1.f});
      }
    }

    // CTA reduction (fixed tree) and the per-token epilogue on thread 0
    if (ENT) {
      const MS3 w = warp_ms3<false>(MS3{acc.m, acc.s, acc_s2});
      if (lane == 0) { sh_m[warp] = w.m; sh_s[warp] = w.s; sh_s2[warp] = w.s2; }
    } else {
      MS w = warp_ms(acc);
      if (lane == 0) { sh_m[warp] = w.m; sh_s[warp] = w.s; }
    }
    __syncthreads();
    if (warp == 0) {
      MS v;
      float ez = 0.f;
      if (ENT) {
        MS3 v3 = lane < NW ? MS3{sh_m[lane], sh_s[lane], sh_s2[lane]} : MS3{-INFINITY, 0.f, 0.f};
        v3 = warp_ms3<false>(v3);
        v = MS{v3.m, v3.s};
        ez = v3.s2 / v3.s;
      } else {
        v = lane < NW ? MS{sh_m[lane], sh_s[lane]} : MS{-INFINITY, 0.f};
        v = warp_ms(v);
      }
      if (lane == 0) {
        const float ls = logf(v.s);
        const float lse = v.m + ls;
        const float sc = (TERMS & kTermsWeight) ? a.scale * tm.w : a.scale;
        // log p_y = (z_y - max) - log(sum): the difference of two logits is exact, so there is no
        // cancellation at any magnitude
        TokenOut o = token_epilogue((ybad ? __int_as_float(0x7fc00000) : zy - v.m) - ls, fabsf(lse) <= kLseMax,
                                    a.old_logp != nullptr, tm.old, tm.A, a.eps, sc);
        if (TERMS & kTermsReg) apply_terms(o, sc, a.kl_kind, a.kl_coef, tm.ref, a.ent_coef, lse - ez);
        a.loss_tok[tm.idx] = o.loss;
        if (a.logp_tok) a.logp_tok[tm.idx] = o.logp;
        if ((TERMS & kTermsReg) && a.entropy_tok) a.entropy_tok[tm.idx] = ENT ? lse - ez : 0.f;
        cnt.tokens++;
        cnt.valid++;
        cnt.clipped += o.clipped;
        cnt.nonfinite += o.nonfinite;
        sh_lse = lse;
        sh_coef = o.coef;
        sh_ez = ez;
      }
    }
    __syncthreads();
    const float lse = sh_lse, coef = sh_coef;
    // entropy gradient: dz_v = p_v (ea + eb z_v) - coef [v == y]
    const float eb = ENT ? ((TERMS & kTermsWeight) ? a.scale * tm.w : a.scale) * a.ent_coef : 0.f;
    const float ea = ENT ? coef - eb * sh_ez : coef;

    // pass 2: dlogits = coef * (softmax - onehot)
    if (dz) {
      uint4* dv = reinterpret_cast<uint4*>(dz);
      if (coef == 0.f && eb == 0.f) {
        const uint4 zero = make_uint4(0, 0, 0, 0);
        for (int64_t j = tid; j < nvec; j += NT) __stcs(dv + j, zero);
        for (int64_t e = tail0 + tid; e < V; e += NT) Vec<T>::store1(dz + e, 0.f);
      } else {
        for (int64_t j = tid; j < nvec; j += NT) {
          float x[VN];
          Vec<T>::unpack(__ldcs(zv + j), x);
#pragma unroll
          for (int i = 0; i < VN; ++i)
            x[i] = ENT ? ent_dz(ex2((x[i] - lse) * kLog2e), x[i], ea, eb) : coef * ex2((x[i] - lse) * kLog2e);
          const int64_t off = (int64_t)y - j * VN;
          if (off >= 0 && off < VN) {
#pragma unroll
            for (int i = 0; i < VN; ++i)
              if (i == off) x[i] -= coef;
          }
          __stcs(dv + j, Vec<T>::pack(x));
        }
        for (int64_t e = tail0 + tid; e < V; e += NT) {
          const float xv = Vec<T>::load1(z + e);
          float p = ENT ? ent_dz(ex2((xv - lse) * kLog2e), xv, ea, eb) : coef * ex2((xv - lse) * kLog2e);
          if (e == y) p -= coef;
          Vec<T>::store1(dz + e, p);
        }
      }
    }
    __syncthreads();  // sh_* are rewritten by the next row
  }
  if (tid == 0) cnt.flush(a.acc);
}

// ------------------------------------------------------------------------------------------
// Cluster kernel: a row is split across the C CTAs of a cluster; CTA r owns the slice
// [r*Vs, r*Vs + n_r) and keeps it in shared memory for both passes. Warp 0 is the producer:
// one lane issues the slice as bulk copies of one chunk each (32 KB, or 16 KB for the
// entropy instances where two CTAs share an SM) into a ring of slots, each completing on its
// own "full" mbarrier, and refills a slot as soon as every consumer warp has released it on
// its "empty" mbarrier. Slots beyond the row's chunks carry the next row's first chunks while
// the current row is exchanged. Warps 1..NCW consume: pass 1 (a log2-domain sum against a lazy
// shift) from shared memory, a fixed-order reduction (shuffle trees within and across warps),
// one cluster barrier per row to exchange (shift, sum) and the target logit through
// distributed shared memory, then pass 2 (dlogits) from shared memory with 16-byte streaming
// stores. HBM sees one read and one write of each row.
// ------------------------------------------------------------------------------------------
constexpr int kMaxChunks = 16;

// Elements of T per 16-byte vector.
template <typename T>
__host__ __device__ constexpr int vec_elems() { return 16 / (int)sizeof(T); }

// Elements per bulk-copied chunk: every consumer thread owns VPT 16-byte vectors of it.
template <typename T>
__host__ __device__ constexpr int cluster_chunk_elems(int NCW, int VPT) { return VPT * NCW * 32 * vec_elems<T>(); }

// A CTA's share of a row, rounded up to whole 16-byte vectors.
template <typename T>
__host__ __device__ constexpr int cluster_slice_elems(int64_t V, int C) {
  return (int)((((V + C - 1) / C) + vec_elems<T>() - 1) / vec_elems<T>() * vec_elems<T>());
}

__host__ __device__ constexpr size_t cluster_tail_bytes(int NCW) {
  return 2 * kMaxChunks * sizeof(uint64_t) + 8 * sizeof(float) + 3 * NCW * sizeof(float) + 16;
}

// Shared memory of the fixed staging buffer (the smallest ring) plus barriers and exchange.
template <typename T>
__host__ __device__ constexpr size_t cluster_smem_bytes(int Vs, int NCW) {
  return ((size_t)Vs * sizeof(T) + 127) / 128 * 128 + cluster_tail_bytes(NCW);
}

// Bounded wait used only when draining after a timeout (ignores the abort flag).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0; i < (1u << 24); ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 255u) == 0 && global_timer_ns() - t0 > 1000000000ull) return;
  }
}

// The elements of one 16-byte vector as floats, written to x[0 .. vec_elems<T>()).
template <typename T>
__device__ __forceinline__ void unpack_at(const uint4& a, float* x) {
  if constexpr (sizeof(T) == 2) {
    x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x); x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
    x[4] = bf16_lo(a.z); x[5] = bf16_hi(a.z); x[6] = bf16_lo(a.w); x[7] = bf16_hi(a.w);
  } else {
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y); x[2] = __uint_as_float(a.z);
    x[3] = __uint_as_float(a.w);
  }
}

// One 16-byte vector of T from floats (round to nearest), the sign of every element flipped
// when NEG.
template <typename T, bool NEG>
__device__ __forceinline__ uint4 pack_vec(const float* x) {
  if constexpr (sizeof(T) == 2) {
    uint4 r = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                         pack_bf16x2(x[6], x[7]));
    if (NEG) {
      r.x ^= 0x80008000u;
      r.y ^= 0x80008000u;
      r.z ^= 0x80008000u;
      r.w ^= 0x80008000u;
    }
    return r;
  } else {
    const uint32_t sg = NEG ? 0x80000000u : 0u;
    return make_uint4(__float_as_uint(x[0]) ^ sg, __float_as_uint(x[1]) ^ sg, __float_as_uint(x[2]) ^ sg,
                      __float_as_uint(x[3]) ^ sg);
  }
}

// The dlogits of one 16-byte vector: (-1)^NEG * 2^(z log2e - cexp), rounded to T (PK: the
// exponent arguments by packed pairs).
template <typename T, bool NEG, bool PK>
__device__ __forceinline__ void dz_vec(const uint4& u, uint4* dst, float cexp) {
  constexpr int E = vec_elems<T>();
  float x[E];
  unpack_at<T>(u, x);
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    if constexpr (PK) {
      const float2 p = ex2_pair(x[i], x[i + 1], cexp);
      x[i] = p.x;
      x[i + 1] = p.y;
    } else {
      x[i] = ex2(fmaf(x[i], kLog2e, -cexp));
      x[i + 1] = ex2(fmaf(x[i + 1], kLog2e, -cexp));
    }
  }
  *dst = pack_vec<T, NEG>(x);  // a plain store: on this GPU faster than an evict-first one here
}

// The dlogits of one vector with the entropy term: 2^(z log2e - lse2) * (ea + eb z), rounded
// to T. GUARD: an element without mass (a -inf logit) gives 0 instead of 0 * inf; needed only
// where pass 1 met such an element.
template <typename T, bool GUARD>
__device__ __forceinline__ void dz_vec_ent(const uint4& u, uint4* dst, float lse2, float ea, float eb) {
  constexpr int E = vec_elems<T>();
  float x[E];
  unpack_at<T>(u, x);
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    const float2 p = ex2_pair(x[i], x[i + 1], lse2);
    if constexpr (GUARD) {
      x[i] = ent_dz(p.x, x[i], ea, eb);
      x[i + 1] = ent_dz(p.y, x[i + 1], ea, eb);
    } else {
      const float2 q = __fmul2_rn(p, __ffma2_rn(make_float2(x[i], x[i + 1]), make_float2(eb, eb), make_float2(ea, ea)));
      x[i] = q.x;
      x[i + 1] = q.y;
    }
  }
  *dst = pack_vec<T, false>(x);
}

// The shared-memory ring: S slots of one chunk each. A CTA's chunks, in row order, take slots
// 0, 1, ..., S-1, 0, ...; the slot's phase bit flips at every wrap. With S equal to the
// chunks of a row every row starts at slot 0 (a fixed staging buffer); with S larger, the
// producer fills the spare slots with the first chunks of the next row while this row is
// still being reduced and exchanged.
struct RingCursor {
  int slot;
  uint32_t ph;
  __device__ __forceinline__ void step(int S) {
    if (++slot == S) {
      slot = 0;
      ph ^= 1u;
    }
  }
  __device__ __forceinline__ void skip(int n, int S) {
    slot += n;
    if (slot >= S) {
      slot -= S;
      ph ^= 1u;
    }
  }
};

// Pass 2 with the entropy term over the CTA's slice, chunk k read from its ring slot.
template <typename T, bool GUARD, int NC, int VPT, int CH>
__device__ __forceinline__ void pass2_slice_ent(const T* ring, RingCursor c, int S, uint4* dz, int n_r,
                                                int nch, int ct, int lane, float lse2, float ea, float eb,
                                                uint64_t* empty) {
  for (int k = 0; k < nch; ++k) {
    constexpr int E = vec_elems<T>();
    const int nv = min(CH, n_r - k * CH) / E;
    const uint4* sv = reinterpret_cast<const uint4*>(ring + (size_t)c.slot * CH);
    uint4* dv = dz + k * (CH / E);
    if (nv == VPT * NC) {
#pragma unroll
      for (int j = 0; j < VPT; ++j) dz_vec_ent<T, GUARD>(sv[ct + j * NC], dv + ct + j * NC, lse2, ea, eb);
    } else {
      for (int v = ct; v < nv; v += NC) dz_vec_ent<T, GUARD>(sv[v], dv + v, lse2, ea, eb);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[c.slot]);
    c.step(S);
  }
}

// Pass 2 over the CTA's slice; each warp releases a chunk's slot once it is done with it.
template <typename T, bool NEG, int NC, int VPT, int CH, bool PK>
__device__ __forceinline__ void pass2_slice(const T* ring, RingCursor c, int S, uint4* dz, int n_r,
                                            int nch, int ct, int lane, float cexp, uint64_t* empty) {
  for (int k = 0; k < nch; ++k) {
    constexpr int E = vec_elems<T>();
    const int nv = min(CH, n_r - k * CH) / E;
    const uint4* sv = reinterpret_cast<const uint4*>(ring + (size_t)c.slot * CH);
    uint4* dv = dz + k * (CH / E);
    if (nv == VPT * NC) {
#pragma unroll
      for (int j = 0; j < VPT; ++j) dz_vec<T, NEG, PK>(sv[ct + j * NC], dv + ct + j * NC, cexp);
    } else {
      for (int v = ct; v < nv; v += NC) dz_vec<T, NEG, PK>(sv[v], dv + v, cexp);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[c.slot]);
    c.step(S);
  }
}

// First row at or after `row` (stepping by `stride`) that is read: not padding and mask = 1.
__device__ __forceinline__ int64_t next_read_row(const RowArgs& a, int64_t row, int64_t stride) {
  for (; row < a.T; row += stride) {
    const int64_t src = row_src(a, row);
    if (src >= 0 && a.mask[src] != 0) return row;
  }
  return a.T;
}

// Bytes of the ring for a slice of Vs elements of T and S slots of CH elements (S no larger
// than the slice's chunk count: the fixed staging buffer, whose last slot is only as long as
// the slice's last chunk).
template <typename T>
__host__ __device__ constexpr size_t cluster_ring_bytes(int Vs, int CH, int S) {
  return S > (Vs + CH - 1) / CH ? (size_t)S * CH * sizeof(T) : ((size_t)Vs * sizeof(T) + 127) / 128 * 128;
}

template <typename T, int C, int NCW, int VPT, int MINB, bool ENT, int TERMS>
__global__ void __launch_bounds__((NCW + 1) * 32, MINB) row_cluster_kernel(RowArgs a, int Vs, int S) {
  constexpr int NC = NCW * 32;
  constexpr int E = vec_elems<T>();  // elements per 16-byte vector
  constexpr int WS = ENT ? 3 : 2;  // floats per warp partial
  // packed two-lane arithmetic, except in the KL instances, whose 32 KB chunks leave no
  // registers for the aligned pairs they need
  constexpr bool PK = !((TERMS & kTermsReg) && !ENT);
  constexpr int CH = cluster_chunk_elems<T>(NCW, VPT);
  extern __shared__ __align__(128) uint8_t smem[];
  const int ring_bytes = (int)cluster_ring_bytes<T>(Vs, CH, S);
  T* ring = reinterpret_cast<T*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ring_bytes);
  uint64_t* empty = full + kMaxChunks;
  float* xch = reinterpret_cast<float*>(empty + kMaxChunks);  // [2 rows][m, s, z_y, s2]
  float* wpart = xch + 8;                                      // [NCW][m, s, s2]
  volatile int* s_abort = reinterpret_cast<volatile int*>(wpart + 3 * NCW);

  const uint32_t rank = cluster_ctarank();
  const int64_t cid = blockIdx.x / C, ncl = gridDim.x / C;
  const int64_t V = a.V;
  const int64_t base = (int64_t)rank * Vs;
  const int n_r = (int)max((int64_t)0, min((int64_t)Vs, V - base));
  const int nch = (n_r + CH - 1) / CH;
  const bool ring_mode = S > (Vs + CH - 1) / CH;
  const int SL = ring_mode ? S : max(nch, 1);      // slots this CTA cycles through
  const int P = ring_mode ? min(S - nch, nch) : 0;  // next-row chunks issued before this row's exchange
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int k = 0; k < kMaxChunks; ++k) {
      mbar_init(&full[k], 1);
      mbar_init(&empty[k], NCW);
    }
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  cluster_sync_all();

  const T* lg = static_cast<const T*>(a.logits);
  T* dg = static_cast<T*>(a.dlogits);
  const uint4 zero = make_uint4(0, 0, 0, 0);
  Counts cnt;
  uint32_t issued = 0;  // producer: chunks issued so far (slot reuse starts at SL)

  if (warp == 0) {
    // ---- producer: one lane issues the bulk copies; the warp joins one exchange per read row ----
    RingCursor pc{0, 0u};
    bool stop = false;  // a wait gave up: issue nothing more
    auto issue = [&](int64_t row, int k) {
      if (stop) return;
      if (issued >= (uint32_t)SL && !mbar_wait_bounded(&empty[pc.slot], pc.ph ^ 1u, s_abort)) {
        stop = true;
        return;
      }
      const int n_k = min(CH, n_r - k * CH);
      mbar_arrive_expect_tx(&full[pc.slot], (uint32_t)n_k * (uint32_t)sizeof(T));
      bulk_g2s(ring + (size_t)pc.slot * CH, lg + row * a.ld + base + (int64_t)k * CH, (uint32_t)n_k * (uint32_t)sizeof(T),
               &full[pc.slot]);
      ++issued;
      pc.step(SL);
    };
    int64_t cur = lane == 0 ? next_read_row(a, cid, ncl) : 0;
    cur = __shfl_sync(0xffffffffu, cur, 0);
    int pre = 0;  // chunks of `cur` issued during the previous row
    while (cur < a.T) {
      int64_t nxt = 0;
      if (lane == 0) {
        for (int k = pre; k < nch; ++k) issue(cur, k);
        nxt = next_read_row(a, cur + ncl, ncl);
        // the spare slots were released by the previous row's pass 2, which the consumers
        // finish before this row's exchange: these waits cannot hold up the exchange
        if (nxt < a.T)
          for (int k = 0; k < P; ++k) issue(nxt, k);
      }
      nxt = __shfl_sync(0xffffffffu, nxt, 0);
      cluster_sync_all();  // this row's exchange
      pre = P;
      cur = nxt;
    }
  } else {
    // ---- consumers ----
    const int ct = tid - 32;
    RingCursor rc{0, 0u};  // slot of the current row's first chunk
    uint32_t vi = 0;       // rows read so far: selects the exchange buffer
    MetaPipe<TERMS> pipe(a, cid, ncl);
    for (int64_t row = cid; row < a.T; row += ncl) {
      const auto tm = pipe.advance(row);
      uint4* dz = dg ? reinterpret_cast<uint4*>(dg + row * a.ld_out + base) : nullptr;
      if (!tm.valid) {
        // masked or padding row: nothing read, nothing exchanged; zero dlogits slice
        if (dz)
          for (int v = ct; v < n_r / E; v += NC) dz[v] = zero;
        if (rank == 0 && ct == 0) {
          cnt.tokens++;
          if (tm.idx >= 0) {
            a.loss_tok[tm.idx] = 0.f;
            if (a.logp_tok) a.logp_tok[tm.idx] = 0.f;
            if ((TERMS & kTermsReg) && a.entropy_tok) a.entropy_tok[tm.idx] = 0.f;
          }
        }
        continue;
      }
      float* xb = xch + 4 * (vi & 1u);
      const int32_t y = tm.y;
      const bool ybad = y < 0 || (int64_t)y >= V;

      // pass 1: log2-domain (shift, sum) over the slice, chunk by chunk as it lands
      MS acc{-INFINITY, 0.f};
      MS3 acc3{-INFINITY, 0.f, 0.f};
      bool guarded = false;  // entropy: pass 1 met a -inf logit among this thread's elements
      RingCursor c = rc;
      for (int k = 0; k < nch; ++k) {
        mbar_wait_bounded(&full[c.slot], c.ph, s_abort);
        const int nv = min(CH, n_r - k * CH) / E;
        const uint4* sv = reinterpret_cast<const uint4*>(ring + (size_t)c.slot * CH);
        if (nv == VPT * NC) {  // full chunk: exactly VPT 16-byte vectors per consumer thread
          float x[VPT * E];
#pragma unroll
          for (int j = 0; j < VPT; ++j) unpack_at<T>(sv[ct + j * NC], x + E * j);
          if (ENT) {
            // blocks of at most 16: the pair sums of a whole 32-element chunk would not stay
            // in registers
            constexpr int EB = VPT * E < 16 ? VPT * E : 16;
#pragma unroll
            for (int h = 0; h < VPT * E / EB; ++h)
              lazy_online3<EB>(acc3, *reinterpret_cast<const float(*)[EB]>(x + EB * h), guarded);
          } else
            lazy_online2<VPT * E, PK>(acc, x);
        } else {
          for (int v = ct; v < nv; v += NC) {
            float x[E];
            unpack_at<T>(sv[v], x);
            if (ENT)
              lazy_online3<E>(acc3, x, guarded);
            else
              lazy_online2<E, PK>(acc, x);
          }
        }
        c.step(SL);
      }
      if (ENT) {
        const MS3 w = warp_ms3<true>(acc3);
        if (lane == 0) {
          wpart[WS * (warp - 1)] = w.m;
          wpart[WS * (warp - 1) + 1] = w.s;
          wpart[WS * (warp - 1) + 2] = w.s2;
        }
      } else {
        const MS w = warp_ms2(acc);
        if (lane == 0) {
          wpart[WS * (warp - 1)] = w.m;
          wpart[WS * (warp - 1) + 1] = w.s;
        }
      }
      named_bar_sync(1, NC);
      if (warp == 1) {
        // the CTA's NCW warp partials combined by a fixed pairwise tree across warp 1's lanes
        MS3 t{-INFINITY, 0.f, 0.f};
        if (ENT) {
          t = group_tree_ms3<NCW>(lane < NCW ? MS3{wpart[WS * lane], wpart[WS * lane + 1], wpart[WS * lane + 2]}
                                             : MS3{-INFINITY, 0.f, 0.f});
        } else {
          const MS t2 = group_tree_ms2<NCW>(lane < NCW ? MS{wpart[WS * lane], wpart[WS * lane + 1]}
                                                       : MS{-INFINITY, 0.f});
          t = MS3{t2.m, t2.s, 0.f};
        }
        if (lane == 0) {
          xb[0] = t.m;
          xb[1] = t.s;
          if (ENT) xb[3] = t.s2;
          if (!ybad && (int64_t)y >= base && (int64_t)y < base + n_r) {
            const int off = (int)((int64_t)y - base), k = off / CH;
            RingCursor cy = rc;
            cy.skip(k, SL);
            xb[2] = Vec<T>::load1(ring + (size_t)cy.slot * CH + (off - k * CH));
          }
        }
      }
      cluster_sync_all();

      // every consumer combines the C slices in rank order: identical LSE in every CTA
      MS tot{-INFINITY, 0.f};
      MS3 tot3{-INFINITY, 0.f, 0.f};
      float zy = __int_as_float(0x7fc00000);
      const uint32_t xaddr = smem_u32(xb);
#pragma unroll
      for (int r = 0; r < C; ++r) {
        const uint32_t ra = mapa_u32(xaddr, (uint32_t)r);
        if (ENT)
          tot3 = ms3_combine2(tot3, MS3{ld_dsmem_f32(ra), ld_dsmem_f32(ra + 4), ld_dsmem_f32(ra + 12)});
        else
          tot = ms2_combine(tot, MS{ld_dsmem_f32(ra), ld_dsmem_f32(ra + 4)});
        if (!ybad && (int64_t)y >= (int64_t)r * Vs && (int64_t)y < (int64_t)(r + 1) * Vs)
          zy = ld_dsmem_f32(ra + 8);
      }
      if (ENT) tot = MS{tot3.m, tot3.s};
      const float l2s = log2f(tot.s);
      const float lse2 = tot.m + l2s;  // log2(sum_v 2^(z_v log2 e)) = LSE * log2(e)
      const float ez = ENT ? tot3.s2 / tot3.s : 0.f;  // sum_v p_v z_v
      const float sc = (TERMS & kTermsWeight) ? a.scale * tm.w : a.scale;
      // log2 p_y = (z_y log2e - m) - log2(sum): one rounding of z_y log2e - m, no cancellation
      TokenOut o = token_epilogue((fmaf(zy, kLog2e, -tot.m) - l2s) * kLn2, fabsf(lse2) <= kLseMax * kLog2e,
                                  a.old_logp != nullptr, tm.old, tm.A, a.eps, sc);
      if (TERMS & kTermsReg) apply_terms(o, sc, a.kl_kind, a.kl_coef, tm.ref, a.ent_coef, lse2 * kLn2 - ez);
      if (rank == 0 && ct == 0) {
        a.loss_tok[tm.idx] = o.loss;
        if (a.logp_tok) a.logp_tok[tm.idx] = o.logp;
        if ((TERMS & kTermsReg) && a.entropy_tok) a.entropy_tok[tm.idx] = ENT ? lse2 * kLn2 - ez : 0.f;
        cnt.tokens++;
        cnt.valid++;
        cnt.clipped += o.clipped;
        cnt.nonfinite += o.nonfinite;
      }
      const float coef = o.coef;
      const float eb = ENT ? sc * a.ent_coef : 0.f;
      if (ENT && dz && eb != 0.f) {
        // with the entropy term: dz_v = p_v (ea + eb z_v) - coef [v == y]
        const float ea = coef - eb * ez;
        // pass 2 visits this thread's pass-1 elements; the warp takes the guarded form if any
        // of its threads met a -inf logit
        if (__any_sync(0xffffffffu, guarded))
          pass2_slice_ent<T, true, NC, VPT, CH>(ring, rc, SL, dz, n_r, nch, ct, lane, lse2, ea, eb, empty);
        else
          pass2_slice_ent<T, false, NC, VPT, CH>(ring, rc, SL, dz, n_r, nch, ct, lane, lse2, ea, eb, empty);
        const int64_t yl = ybad ? -1 : (int64_t)y - base;
        if (yl >= 0 && yl < n_r && ct == (int)(((yl / E) % (CH / E)) % NC)) {
          const float dzy = ent_dz(ex2(fmaf(zy, kLog2e, -lse2)), zy, ea, eb) - coef;
          Vec<T>::store1(reinterpret_cast<T*>(dz) + yl, dzy);
        }
      } else if (dz && coef != 0.f) {
        // pass 2: |coef| * softmax = 2^(z log2e - (lse2 - log2|coef|)), the sign applied to
        // the packed bf16 pairs; the target element coef * (p_y - 1) is written on its own
        const float cexp = lse2 - log2f(fabsf(coef));
        if (coef < 0.f)
          pass2_slice<T, true, NC, VPT, CH, PK>(ring, rc, SL, dz, n_r, nch, ct, lane, cexp, empty);
        else
          pass2_slice<T, false, NC, VPT, CH, PK>(ring, rc, SL, dz, n_r, nch, ct, lane, cexp, empty);
        // the target element overwrites what the vector pass wrote (same thread, program order)
        const int64_t yl = ybad ? -1 : (int64_t)y - base;
        if (yl >= 0 && yl < n_r && ct == (int)(((yl / E) % (CH / E)) % NC)) {
          const float dzy = coef * ex2(fmaf(zy, kLog2e, -lse2)) - coef;
          Vec<T>::store1(reinterpret_cast<T*>(dz) + yl, dzy);
        }
      } else {
        if (dz)
          for (int v = ct; v < n_r / E; v += NC) dz[v] = zero;
        __syncwarp();
        if (lane == 0) {
          RingCursor ce = rc;
          for (int k = 0; k < nch; ++k) {
            mbar_arrive(&empty[ce.slot]);
            ce.step(SL);
          }
        }
      }
      rc.skip(nch, SL);
      ++vi;
    }
  }

  __syncthreads();
  if (*s_abort) {
    // a wait gave up: let every copy still in flight land before the CTA's memory goes away
    // (the last use of slot s is copy number issued-1-s counted back in steps of SL)
    if (tid == 0)
      for (int sl = 0; sl < SL && (uint32_t)sl < issued; ++sl)
        mbar_drain(&full[sl], ((issued - 1u - (uint32_t)sl) / (uint32_t)SL) & 1u);
    if (tid == 0) atomicOr(&a.acc->flags, kFlagWaitTimeout);
  }
  cluster_sync_all();  // no CTA leaves while a peer may still read its exchange slots
  if (tid == 32 && rank == 0) cnt.flush(a.acc);
}

// ------------------------------------------------------------------------------------------
// Forward-only cluster kernel (no dlogits, no extra terms): the pi_old ahead pass. It splits
// rows, chunks them and assigns elements to threads exactly as row_cluster_kernel<T, C, NCW,
// VPT> does, and combines the partial sums in the same order, so the log-prob, the loss and
// the counts are the same bits. What differs is that no consumer waits for a row's exchange:
//  * each consumer warp releases a chunk's slot as soon as it has folded the chunk in, and the
//    producer streams the cluster's rows through the ring with no per-row barrier;
//  * each consumer warp sends its (shift, sum) straight into CTA 0's exchange buffer with an
//    asynchronous DSMEM store that completes on CTA 0's mbarrier, and goes on to the next row
//    without a fence;
//  * a combiner warp of CTA 0 (the block's last warp) takes the rows in order, combines each
//    row's C * NCW partials (warps in order within a CTA, then CTAs in rank order) and writes
//    the token's outputs; it also writes the outputs of masked and padding rows.
// kFwdBufs exchange buffers, each handed back by the combiner through an mbarrier in every
// CTA, bound how far a consumer can run ahead of the combines.
// ------------------------------------------------------------------------------------------
constexpr int kFwdBufs = 4;

__host__ __device__ constexpr size_t fwd_tail_bytes(int C, int NCW) {
  return (2 * kMaxChunks + 2 * kFwdBufs) * sizeof(uint64_t) + (size_t)kFwdBufs * C * NCW * 2 * sizeof(float) +
         kFwdBufs * sizeof(float) + 16;
}

// Threads per block of the forward-only kernel: producer, NCW consumers, combiner.
__host__ __device__ constexpr int fwd_block_threads(int NCW) { return (NCW + 2) * 32; }

// First row at or after `from` (stepping by `stride`) that is read, examining 32 rows at once;
// every lane of the warp calls it and gets the same answer.
__device__ __forceinline__ int64_t scan_read_row(const RowArgs& a, int64_t from, int64_t stride, int lane) {
  for (; from < a.T; from += 32 * stride) {
    const int64_t r = from + (int64_t)lane * stride;
    bool ok = false;
    if (r < a.T) {
      const int64_t src = row_src(a, r);
      ok = src >= 0 && a.mask[src] != 0;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (bal) return from + (int64_t)(__ffs(bal) - 1) * stride;
  }
  return a.T;
}

template <typename T, int C, int NCW, int VPT>
__global__ void __launch_bounds__(fwd_block_threads(NCW), 1) row_fwd_kernel(RowArgs a, int Vs, int S) {
  constexpr int NC = NCW * 32;
  constexpr int E = vec_elems<T>();
  constexpr int CH = cluster_chunk_elems<T>(NCW, VPT);
  constexpr int NP = C * NCW;  // partials per row
  constexpr bool PK = true;
  extern __shared__ __align__(128) uint8_t smem[];
  T* ring = reinterpret_cast<T*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)S * CH * sizeof(T));
  uint64_t* empty = full + kMaxChunks;
  uint64_t* xfull = empty + kMaxChunks;  // CTA 0: all partials of the buffer's row are in
  uint64_t* xempty = xfull + kFwdBufs;   // every CTA: CTA 0 has read the buffer
  float* part = reinterpret_cast<float*>(xempty + kFwdBufs);  // CTA 0: [buffer][C * NCW][m, s]
  float* zyv = part + kFwdBufs * NP * 2;                      // CTA 0: [buffer] target logit
  volatile int* s_abort = reinterpret_cast<volatile int*>(zyv + kFwdBufs);

  const uint32_t rank = cluster_ctarank();
  const int64_t cid = blockIdx.x / C, ncl = gridDim.x / C;
  const int64_t V = a.V;
  const int64_t base = (int64_t)rank * Vs;
  const int n_r = (int)max((int64_t)0, min((int64_t)Vs, V - base));
  const int nch = (n_r + CH - 1) / CH;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int k = 0; k < kMaxChunks; ++k) {
      mbar_init(&full[k], 1);
      mbar_init(&empty[k], NCW);
    }
    for (int b = 0; b < kFwdBufs; ++b) {
      mbar_init(&xfull[b], 1);  // the combiner's arrive, plus the bytes of the row's stores
      mbar_init(&xempty[b], 1);
    }
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  cluster_sync_all();

  const T* lg = static_cast<const T*>(a.logits);
  Counts cnt;
  uint32_t issued = 0;  // producer: chunks issued so far (slot reuse starts at S)

  if (warp == 0) {
    // ---- producer: lane 0 streams the read rows' chunks; the warp looks for the next row ----
    RingCursor pc{0, 0u};
    int64_t cur = scan_read_row(a, cid, ncl, lane);
    while (cur < a.T) {
      // the next 32 candidate rows: their index and mask loads are in flight while lane 0
      // issues this row's copies
      const int64_t cand = cur + (int64_t)(lane + 1) * ncl;
      const int64_t csrc = cand < a.T ? row_src(a, cand) : -1;
      bool stop = false;
      if (lane == 0) {
        for (int k = 0; k < nch; ++k) {
          if (issued >= (uint32_t)S && !mbar_wait_bounded(&empty[pc.slot], pc.ph ^ 1u, s_abort)) {
            stop = true;
            break;
          }
          const int n_k = min(CH, n_r - k * CH);
          mbar_arrive_expect_tx(&full[pc.slot], (uint32_t)n_k * (uint32_t)sizeof(T));
          bulk_g2s(ring + (size_t)pc.slot * CH, lg + cur * a.ld + base + (int64_t)k * CH,
                   (uint32_t)n_k * (uint32_t)sizeof(T), &full[pc.slot]);
          ++issued;
          pc.step(S);
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) break;  // a wait gave up: issue nothing more
      const bool ok = csrc >= 0 && a.mask[csrc] != 0;
      const unsigned bal = __ballot_sync(0xffffffffu, ok);
      cur = bal ? cur + (int64_t)__ffs(bal) * ncl : scan_read_row(a, cur + 33 * ncl, ncl, lane);
    }
  } else if (warp <= NCW) {
    // ---- consumers ----
    const int ct = tid - 32, cw = warp - 1;
    RingCursor rc{0, 0u};
    uint32_t xi = 0;  // read rows so far: the exchange sequence number
    MetaPipe<0> pipe(a, cid, ncl);
    for (int64_t row = cid; row < a.T; row += ncl) {
      // the row's metadata: lane 0 keeps the prefetch pipeline and broadcasts, so lane 31,
      // which releases the ring slots, has no global load in flight for its release to wait on
      RowMeta<0> tm{};
      if (lane == 0) tm = pipe.advance(row);
      tm.valid = __shfl_sync(0xffffffffu, (int)tm.valid, 0) != 0;
      tm.y = __shfl_sync(0xffffffffu, tm.y, 0);
      if (!tm.valid) continue;  // masked or padding row: nothing read, nothing exchanged
      // where the target logit sits in this CTA's slice, and which thread reads it
      const int64_t yo = (tm.y < 0 || (int64_t)tm.y >= V) ? -1 : (int64_t)tm.y - base;
      const bool own = yo >= 0 && yo < n_r;
      const int ky = own ? (int)(yo / CH) : -1;
      const int oy = own ? (int)(yo - (int64_t)ky * CH) : 0;
      const int cty = (oy / E) % NC;
      float zyl = 0.f;

      // pass 1, slot by slot as the chunks land; each slot is released once folded in
      MS acc{-INFINITY, 0.f};
      for (int k = 0; k < nch; ++k) {
        mbar_wait_bounded(&full[rc.slot], rc.ph, s_abort);
        const int nv = min(CH, n_r - k * CH) / E;
        const uint4* sv = reinterpret_cast<const uint4*>(ring + (size_t)rc.slot * CH);
        if (nv == VPT * NC) {
          float x[VPT * E];
#pragma unroll
          for (int j = 0; j < VPT; ++j) unpack_at<T>(sv[ct + j * NC], x + E * j);
          lazy_online2<VPT * E, PK>(acc, x);
        } else {
          for (int v = ct; v < nv; v += NC) {
            float x[E];
            unpack_at<T>(sv[v], x);
            lazy_online2<E, PK>(acc, x);
          }
        }
        if (k == ky && ct == cty) zyl = Vec<T>::load1(ring + (size_t)rc.slot * CH + oy);
        __syncwarp();
        if (lane == 31) mbar_arrive(&empty[rc.slot]);
        rc.step(S);
      }

      // the warp's partial (and the target logit, from the warp that read it) to CTA 0
      const MS w = warp_ms2(acc);
      const bool wown = own && cty / 32 == cw;
      const float zy = wown ? __shfl_sync(0xffffffffu, zyl, cty & 31) : 0.f;
      if (lane == 0) {
        const uint32_t b = xi % kFwdBufs, u = xi / kFwdBufs;
        // the buffer is free once the combiner's arrive completed this phase. The signal
        // publishes no data (the combiner had consumed what it read from the buffer before
        // arriving), so the wait needs no cluster-scope acquire; one cost the ahead pass 5%.
        if (u > 0) mbar_wait_bounded(&xempty[b], (u - 1u) & 1u, s_abort);
        const uint32_t bar = mapa_u32(smem_u32(&xfull[b]), 0u);
        st_async_v2f32(mapa_u32(smem_u32(part + 2 * (b * NP + rank * NCW + cw)), 0u), w.m, w.s, bar);
        if (wown) st_async_f32(mapa_u32(smem_u32(zyv + b), 0u), zy, bar);
      }
      ++xi;
    }
  } else if (rank == 0) {
    // ---- combiner (CTA 0): every row of the cluster in order; the read rows' log-sum-exp
    // from their partials, then the token's outputs ----
    uint32_t xi = 0;
    MetaPipe<0> pipe(a, cid, ncl);
    for (int64_t row = cid; row < a.T; row += ncl) {
      const auto tm = pipe.advance(row);
      if (!tm.valid) {
        if (lane == 0) {
          cnt.tokens++;
          if (tm.idx >= 0) {
            a.loss_tok[tm.idx] = 0.f;
            if (a.logp_tok) a.logp_tok[tm.idx] = 0.f;
          }
        }
        continue;
      }
      const uint32_t b = xi % kFwdBufs, u = xi / kFwdBufs;
      const bool ybad = tm.y < 0 || (int64_t)tm.y >= V;
      // the phase completes once every warp's partial (and the target logit) has landed.
      // Phase u-1 is complete: this warp waited for it four read rows ago, and no store of
      // this row is issued before the buffer's release that followed that wait. The partials
      // come by st.async, whose bytes the phase's transaction count tracks: observing the
      // phase complete makes them visible, as for a bulk copy into this CTA, so the wait is
      // the CTA-scope one (a cluster-scope acquire here cost the ahead pass another 4%).
      if (lane == 0) mbar_arrive_expect_tx_relaxed(&xfull[b], NP * 8u + (ybad ? 0u : 4u));
      mbar_wait_bounded(&xfull[b], u & 1u, s_abort);
      // each CTA's NCW partials by the general kernel's pairwise tree (32 / NCW CTAs at a time,
      // one per NCW-lane group), then the CTAs in rank order
      constexpr int G = 32 / NCW;
      MS tot{-INFINITY, 0.f};
#pragma unroll
      for (int r0 = 0; r0 < C; r0 += G) {
        const int r = r0 + lane / NCW;
        MS v{-INFINITY, 0.f};
        if (r < C) {
          const float* p = part + 2 * (b * NP + r * NCW + lane % NCW);
          v = MS{p[0], p[1]};
        }
        v = group_tree_ms2<NCW>(v);
#pragma unroll
        for (int k = 0; k < G; ++k)
          if (r0 + k < C)
            tot = ms2_combine(tot, MS{__shfl_sync(0xffffffffu, v.m, k * NCW), __shfl_sync(0xffffffffu, v.s, k * NCW)});
      }
      const float zy = ybad ? __int_as_float(0x7fc00000) : zyv[b];
      __syncwarp();
      if (lane == 0) {
        const float l2s = log2f(tot.s);
        const float lse2 = tot.m + l2s;
        const TokenOut o = token_epilogue((fmaf(zy, kLog2e, -tot.m) - l2s) * kLn2, fabsf(lse2) <= kLseMax * kLog2e,
                                          a.old_logp != nullptr, tm.old, tm.A, a.eps, a.scale);
        // the buffer is free again in every CTA: what was read from it has been consumed
        // (by the shuffles and the epilogue), so the signal needs no fence
        for (int r = 0; r < C; ++r) mbar_arrive_remote_relaxed(mapa_u32(smem_u32(&xempty[b]), (uint32_t)r));
        a.loss_tok[tm.idx] = o.loss;
        if (a.logp_tok) a.logp_tok[tm.idx] = o.logp;
        cnt.tokens++;
        cnt.valid++;
        cnt.clipped += o.clipped;
        cnt.nonfinite += o.nonfinite;
      }
      ++xi;
    }
  }

  __syncthreads();
  if (*s_abort) {
    if (tid == 0)
      for (int sl = 0; sl < S && (uint32_t)sl < issued; ++sl)
        mbar_drain(&full[sl], ((issued - 1u - (uint32_t)sl) / (uint32_t)S) & 1u);
    if (tid == 0) atomicOr(&a.acc->flags, kFlagWaitTimeout);
  }
  cluster_sync_all();  // no CTA leaves while a peer may still store into or arrive on its memory
  if (rank == 0 && warp == NCW + 1 && lane == 0) cnt.flush(a.acc);
}

}  // namespace grpo
