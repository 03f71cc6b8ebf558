// Fused LM-head variant of the loss: the logits z = h W^T are produced on the tensor cores
// tile by tile and consumed by the softmax in the GEMM epilogue; neither the [T, V] logits nor
// their softmax nor any [T, V] matrix derived from them is ever held in memory ("Sizing
// mini-batches and micro-batches", "The problem": the log-softmax over the vocabulary of
// 2048-token completions is what runs out of memory).
//
//  pass A     tcgen05 GEMM over every (256-token x 256-vocabulary) tile; the epilogue reduces
//             each token's tile to a log2-domain (shift, sum-exp) partial and picks up the
//             target logit.
//  reduce     per token: combine the partials in a fixed order -> LSE, log-prob, ratio,
//             clipped surrogate, gradient coefficient (the row pass's token epilogue).
//  partition  the live tokens (a dlogits row that is not all zero) first, in token order; their
//             hidden states gathered into a compact buffer; the others' d_h rows zeroed. The
//             live count stays on the device and sets the backward GEMMs' extents.
//  backward   per vocabulary chunk c (at most 66 tiles, 16896 columns): the same GEMM recomputes
//             the chunk's logits of the live tokens and its epilogue writes their bf16 dlogits
//             dz_c into a bounded [T, chunk] buffer (two buffers, used in turn); then d_h (+)=
//             dz_c W_c and dW_c = dz_c^T h_live, both on the same tcgen05 kernel with float32
//             outputs, on a second stream so that the next chunk's recompute runs beside them.
//             d_h is accumulated over the chunks in chunk order (a fixed order: the result does
//             not depend on how the tokens are split into calls).
//
// All four contractions run on grpo::lmhead::gemm_kernel (grpo_lmhead_gemm.cuh): 2-CTA
// clusters with paired tcgen05.mma (cta_group::2, 256 x 256 tiles), plain TMA tile loads.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "grpo_lmhead_gemm.cuh"

namespace grpo {
namespace lmhead {

// Inputs and outputs of the per-token reduce.
struct ReduceArgs {
  int64_t T, V;
  int n_col_tiles;
  const float *part_m, *part_s, *part_s2, *zy;  // part_s2: entropy instance only
  const int32_t* target;
  const float *old_logp, *adv;
  const uint8_t* mask;
  float eps, scale;
  // terms (TERMS): KL to a reference policy, entropy bonus, per-token weight of the grad scale
  int32_t kl_kind;
  float kl_coef, ent_coef;
  const float *ref_logp, *w_tok;
  float* entropy_tok;
  float *lse2_out, *coef_out, *ea_out, *eb_out;  // ea, eb: entropy instance only
  float *loss_tok, *logp_tok;
  grpo_step_acc* acc;
  // when pass A skipped the masked tokens: the compact order (valid tokens first) and the
  // valid count; NULL otherwise
  const int32_t *idx, *live_n;
};

// Per token: combine the vocabulary-tile partials, then the token epilogue. A block takes 32
// tokens (lane = token, so every partial load is one coalesced 128-byte line) and its 8 warps
// split the tiles: warp w folds tiles w, w + 8, ... in order; warp 0 then folds the 8 warp
// partials in warp order. The order depends only on the tile count. ENT: the partials carry
// sum e z, and the token's entropy LSE - E_p[z] is formed; TERMS: the regularisers and the
// per-token weight are applied as in the row pass.
constexpr int kReduceWarps = 8;

template <bool ENT, bool TERMS>
__global__ void __launch_bounds__(kReduceWarps * 32) reduce_kernel(ReduceArgs a) {
  __shared__ float wm[kReduceWarps][32], ws[kReduceWarps][32], ws2[kReduceWarps][32];
  __shared__ unsigned long long sc[4];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x < 4) sc[threadIdx.x] = 0;
  // i: this lane's row of the partials (a token, or a row of the compact order when pass A
  // skipped the masked tokens); tok: the token whose inputs and outputs it holds
  const int64_t T = a.T, i = (int64_t)blockIdx.x * 32 + lane;
  const int64_t tok = (a.idx && i < T) ? (int64_t)a.idx[i] : i;
  const bool live = i < T && (a.idx ? i < (int64_t)*a.live_n : a.mask[i] != 0);
  MS3 t{-INFINITY, 0.f, 0.f};
  if (live) {
#pragma unroll 4
    for (int c = w; c < a.n_col_tiles; c += kReduceWarps) {
      const int64_t k = (int64_t)c * T + i;
      if (ENT) {
        t = ms3_combine2(t, MS3{a.part_m[k], a.part_s[k], a.part_s2[k]});
      } else {
        const MS u = ms2_combine(MS{t.m, t.s}, MS{a.part_m[k], a.part_s[k]});
        t = MS3{u.m, u.s, 0.f};
      }
    }
  }
  wm[w][lane] = t.m;
  ws[w][lane] = t.s;
  if (ENT) ws2[w][lane] = t.s2;
  __syncthreads();
  unsigned long long v_valid = 0, v_clip = 0, v_nf = 0, v_tok = 0;
  if (w == 0 && i < T) {
    v_tok = 1;
    float coef = 0.f, l2 = 0.f, ea = 0.f, eb = 0.f, H = 0.f;
    if (live) {
      MS3 tot{wm[0][lane], ws[0][lane], ENT ? ws2[0][lane] : 0.f};
#pragma unroll
      for (int k = 1; k < kReduceWarps; ++k) {
        if (ENT) {
          tot = ms3_combine2(tot, MS3{wm[k][lane], ws[k][lane], ws2[k][lane]});
        } else {
          const MS u = ms2_combine(MS{tot.m, tot.s}, MS{wm[k][lane], ws[k][lane]});
          tot = MS3{u.m, u.s, 0.f};
        }
      }
      const float l2s = log2f(tot.s);
      l2 = tot.m + l2s;
      const float ez = ENT ? tot.s2 / tot.s : 0.f;  // sum_v p_v z_v
      const int32_t y = a.target[tok];
      const float z = (y >= 0 && (int64_t)y < a.V) ? a.zy[tok] : __int_as_float(0x7fc00000);
      const float scl = (TERMS && a.w_tok) ? a.scale * a.w_tok[tok] : a.scale;
      // log2 p_y = (z_y log2e - m) - log2(sum), without cancellation
      TokenOut o = token_epilogue((fmaf(z, kLog2e, -tot.m) - l2s) * kLn2, fabsf(l2) <= kLseMax * kLog2e,
                                  a.old_logp != nullptr, a.old_logp ? a.old_logp[tok] : 0.f, a.adv[tok], a.eps,
                                  scl);
      H = ENT ? l2 * kLn2 - ez : 0.f;
      if (TERMS)
        apply_terms(o, scl, a.kl_kind, a.kl_coef, a.kl_kind != GRPO_KL_NONE ? a.ref_logp[tok] : 0.f, a.ent_coef,
                    H);
      a.loss_tok[tok] = o.loss;
      if (a.logp_tok) a.logp_tok[tok] = o.logp;
      coef = o.coef;
      if (ENT) {
        eb = a.ent_coef * scl;
        ea = coef - eb * ez;
      }
      v_valid = 1;
      v_clip = o.clipped;
      v_nf = o.nonfinite;
    } else {
      a.loss_tok[tok] = 0.f;
      if (a.logp_tok) a.logp_tok[tok] = 0.f;
    }
    a.lse2_out[tok] = l2;
    a.coef_out[tok] = coef;
    if (ENT) {
      a.ea_out[tok] = ea;
      a.eb_out[tok] = eb;
    }
    if (TERMS && a.entropy_tok) a.entropy_tok[tok] = H;
  }
  if (v_tok) atomicAdd(&sc[0], v_tok);
  if (v_valid) atomicAdd(&sc[1], v_valid);
  if (v_clip) atomicAdd(&sc[2], v_clip);
  if (v_nf) atomicAdd(&sc[3], v_nf);
  __syncthreads();
  if (threadIdx.x == 0) {
    if (sc[0]) atomicAdd(reinterpret_cast<unsigned long long*>(&a.acc->n_tokens), sc[0]);
    if (sc[1]) atomicAdd(reinterpret_cast<unsigned long long*>(&a.acc->n_valid), sc[1]);
    if (sc[2]) atomicAdd(reinterpret_cast<unsigned long long*>(&a.acc->n_clipped), sc[2]);
    if (sc[3]) atomicAdd(reinterpret_cast<unsigned long long*>(&a.acc->n_nonfinite), sc[3]);
  }
}

// The backward's live tokens: those whose dlogits row is not all zero (a nonzero gradient
// coefficient; with the entropy bonus, a nonzero ea or eb). A token with a zero coefficient
// (masked, zero advantage, clipped, and no regulariser) contributes exact zeros to d_h and dW,
// so the backward's three GEMMs run over the live tokens only. One block writes a stable
// partition of the token indices, the live ones first, in token order, and the live count.
// With `mask` non-NULL the partition is by the mask instead (the valid tokens first), for a
// pass A that skips the masked tokens.
constexpr int kPartThreads = 1024;

__global__ void __launch_bounds__(kPartThreads) partition_kernel(int64_t T, const uint8_t* mask, const float* coef,
                                                                 const float* ea, const float* eb, int32_t* idx,
                                                                 int32_t* live_n) {
  __shared__ int32_t warp_sum[kPartThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int64_t per = (T + kPartThreads - 1) / kPartThreads;
  const int64_t b = (int64_t)tid * per, e = b + per < T ? b + per : T;
  auto live = [&](int64_t t) {
    return mask ? mask[t] != 0 : (ea ? (ea[t] != 0.f || eb[t] != 0.f) : coef[t] != 0.f);
  };
  int32_t c = 0;
  for (int64_t t = b; t < e; ++t) c += live(t) ? 1 : 0;
  // exclusive scan of the per-thread counts: within the warp, then over the warp totals
  int32_t x = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sum[w] = x;
  __syncthreads();
  if (w == 0) {
    int32_t v = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    warp_sum[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  const int32_t total = warp_sum[kPartThreads / 32 - 1];
  int32_t pos = (w > 0 ? warp_sum[w - 1] : 0) + x - c;  // live tokens before this thread's range
  for (int64_t t = b; t < e; ++t) {
    if (live(t))
      idx[pos++] = (int32_t)t;
    else
      idx[total + (t - pos)] = (int32_t)t;  // t - pos = dead tokens before t
  }
  if (tid == 0) *live_n = total;
}

// Row i of the compact order, one warp per row: a live token's hidden state is copied into the
// compact buffer; the rows from the live count to the padded count are zeroed (dW reduces over
// them); a dead token's d_h row is zeroed (no GEMM writes it).
__global__ void __launch_bounds__(256) gather_kernel(int64_t T, int H, const __nv_bfloat16* h, const int32_t* idx,
                                                     const int32_t* live_n, __nv_bfloat16* h_live, float* d_h) {
  const int64_t nl = *live_n;
  const int64_t pad = live_pad(nl, T) < T ? live_pad(nl, T) : T;
  const int lane = threadIdx.x & 31;
  const int nvec = H >> 3;  // 16-byte vectors of a bf16 row (H is a multiple of 64)
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < T; i += warps) {
    const int64_t tok = idx[i];
    uint4* dst = reinterpret_cast<uint4*>(h_live) + i * nvec;
    if (i < nl) {
      const uint4* src = reinterpret_cast<const uint4*>(h) + tok * nvec;
      for (int k = lane; k < nvec; k += 32) dst[k] = src[k];
      continue;
    }
    if (i < pad)
      for (int k = lane; k < nvec; k += 32) dst[k] = z4;
    if (d_h) {  // a float row is two 16-byte vectors per bf16 vector
      uint4* row = reinterpret_cast<uint4*>(d_h) + tok * (2 * nvec);
      for (int k = lane; k < 2 * nvec; k += 32) row[k] = z4;
    }
  }
}

// ---- host -------------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 matrix [outer][ld] of which [outer][inner] is addressed, box {64, box_outer}, 128-byte
// swizzle; reads past either extent return zeros.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The dlogits chunk buffer [T][ld] as a TMA store target: the chunk's vc columns, box 32 x 32,
// 64-byte swizzle (the epilogue's staging layout).
bool map_dz_store(CUtensorMap* m, const void* base, int64_t T, int64_t vc, int64_t ld) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)vc, (cuuint64_t)T};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)EPI_BOX, (cuuint32_t)EPI_BOX};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand maps. K-major [rows][K]: box {64 K, box_rows rows}. MN-major [K][MN]: box {64 MN, 64 K}.
bool map_k(CUtensorMap* m, const void* base, int64_t rows, int64_t k, int64_t ld, int box_rows) {
  return make_map(m, base, (uint64_t)k, (uint64_t)rows, (uint64_t)ld, (uint32_t)box_rows);
}
bool map_mn(CUtensorMap* m, const void* base, int64_t k, int64_t mn, int64_t ld) {
  return make_map(m, base, (uint64_t)mn, (uint64_t)k, (uint64_t)ld, 64u);
}

// CTAs per tile: 2 (paired MMA, the default) or 1 (GRPO_LMHEAD_CTA_GROUP=1, kept for comparison).
int cta_group() {
  const char* e = getenv("GRPO_LMHEAD_CTA_GROUP");
  return (e && e[0] == '1') ? 1 : 2;
}

// One persistent launch over g's units. The first launch of an instance on a device sets its
// shared-memory limit and caches how many CTAs (or CTA pairs) fit at once.
template <int CG, int EPI, bool AMN, bool BMN>
int launch_t(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc, GemmArgs g, cudaStream_t st) {
  using S = Shape<CG, EPI>;
  auto kern = gemm_kernel<CG, EPI, AMN, BMN>;
  g.n_m = (int)((g.M + BM * CG - 1) / (BM * CG));
  int dev = 0;
  GRPO_CUDA_TRY(cudaGetDevice(&dev));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = S::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = CG == 2 ? 1 : 0;
  int max_units = 0;
  {
    static std::mutex mu;
    static int cached[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64) max_units = cached[dev];
    if (max_units == 0) {
      GRPO_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM));
      if (CG == 2) {
        cfg.gridDim = dim3(2 * 1024, 1, 1);
        GRPO_CUDA_TRY(cudaOccupancyMaxActiveClusters(&max_units, kern, &cfg));
      } else {
        max_units = sm_count();
      }
      if (max_units < 1) return GRPO_ERR_UNSUPPORTED;
      if (dev >= 0 && dev < 64) cached[dev] = max_units;
    }
  }
  const int64_t units = std::min<int64_t>((int64_t)g.n_m * g.n_n, max_units);
  if (units <= 0) return GRPO_OK;
  cfg.gridDim = dim3((unsigned)(CG * units), 1, 1);
  GRPO_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, g));
  return GRPO_OK;
}

// mc: the TMA store target of the dlogits epilogue (unused by the other epilogues)
template <int EPI, bool AMN, bool BMN>
int launch(int cg, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc, const GemmArgs& g,
           cudaStream_t st) {
  return cg == 2 ? launch_t<2, EPI, AMN, BMN>(ma, mb, mc, g, st) : launch_t<1, EPI, AMN, BMN>(ma, mb, mc, g, st);
}

// Logits GEMM over vocabulary tiles [col_tile0, col_tile0 + g.n_n): A = h [T, H], B = W [V, H],
// both K-major; the epilogue is EPI.
template <int EPI>
int logits_gemm(int cg, const void* h, const void* W, int64_t T, int64_t V, int64_t H, GemmArgs g,
                cudaStream_t st, int64_t vc = 0) {
  CUtensorMap ma, mb, mc = {};
  if (!map_k(&ma, h, T, H, H, BM) || !map_k(&mb, W, V, H, H, BN / cg)) return GRPO_ERR_UNSUPPORTED;
  if (EPI == EPI_DLOGITS && !map_dz_store(&mc, g.dz, T, vc, g.ldz)) return GRPO_ERR_UNSUPPORTED;
  g.M = T;
  g.K = H;
  g.V = V;
  g.m_fast = 1;  // consecutive units share the W tile
  return launch<EPI, false, false>(cg, ma, mb, mc, g, st);
}

}  // namespace lmhead
}  // namespace grpo

using namespace grpo;
using namespace grpo::lmhead;

namespace {

// Vocabulary tiles per backward chunk: at most 66 (16896 columns), the chunks of equal width
// (V = 151936 -> 594 tiles -> 9 chunks of 66).
constexpr int kMaxChunkTiles = 66;

struct WsLayout {
  // dz, dz2: the two dlogits chunk buffers; then (after the forward pass's prefix) part_s2,
  // ea, eb: the entropy bonus's third partial and its per-token coefficients; idx, live_n,
  // h_live: the backward's token partition, live count and compact hidden states
  size_t part_m, part_s, zy, lse2, coef, dz, dz2, part_s2, ea, eb, idx, live_n, h_live, total;
  int n_col_tiles, chunk_tiles;
  int64_t vchunk;  // columns of the dlogits chunk buffer
};

WsLayout ws_layout(int64_t T, int64_t V, int64_t H) {
  WsLayout w{};
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  w.n_col_tiles = (int)((V + BN - 1) / BN);
  const int n_chunks = (w.n_col_tiles + kMaxChunkTiles - 1) / kMaxChunkTiles;
  w.chunk_tiles = (w.n_col_tiles + n_chunks - 1) / n_chunks;
  w.vchunk = (int64_t)w.chunk_tiles * BN;
  size_t off = 0;
  w.part_m = off; off += up((size_t)w.n_col_tiles * T * 4);
  w.part_s = off; off += up((size_t)w.n_col_tiles * T * 4);
  w.zy = off; off += up((size_t)T * 4);
  w.lse2 = off; off += up((size_t)T * 4);
  w.coef = off; off += up((size_t)T * 4);
  w.dz = off; off += up((size_t)T * w.vchunk * 2);
  w.dz2 = off; off += up((size_t)T * w.vchunk * 2);
  w.part_s2 = off; off += up((size_t)w.n_col_tiles * T * 4);
  w.ea = off; off += up((size_t)T * 4);
  w.eb = off; off += up((size_t)T * 4);
  w.idx = off; off += up((size_t)T * 4);
  w.live_n = off; off += up(4);
  w.h_live = off; off += up((size_t)T * H * 2);
  w.total = off;
  return w;
}

struct Scratch {
  float *part_m, *part_s, *zy, *lse2, *coef;
  __nv_bfloat16* dz[2];
  // NULL when the region lies past the scratch (the no-alloc forward)
  float *part_s2, *ea, *eb;
  int32_t *idx, *live_n;
  __nv_bfloat16* h_live;
};

// The regions of a workspace: all of them (full), or only the forward pass's prefix.
Scratch carve(void* base, const WsLayout& ws, bool full) {
  uint8_t* b = static_cast<uint8_t*>(base);
  Scratch s{reinterpret_cast<float*>(b + ws.part_m), reinterpret_cast<float*>(b + ws.part_s),
            reinterpret_cast<float*>(b + ws.zy),     reinterpret_cast<float*>(b + ws.lse2),
            reinterpret_cast<float*>(b + ws.coef),   {nullptr, nullptr},
            nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  if (full) {
    s.dz[0] = reinterpret_cast<__nv_bfloat16*>(b + ws.dz);
    s.dz[1] = reinterpret_cast<__nv_bfloat16*>(b + ws.dz2);
    s.part_s2 = reinterpret_cast<float*>(b + ws.part_s2);
    s.ea = reinterpret_cast<float*>(b + ws.ea);
    s.eb = reinterpret_cast<float*>(b + ws.eb);
    s.idx = reinterpret_cast<int32_t*>(b + ws.idx);
    s.live_n = reinterpret_cast<int32_t*>(b + ws.live_n);
    s.h_live = reinterpret_cast<__nv_bfloat16*>(b + ws.h_live);
  }
  return s;
}

// Whether a call's terms need the entropy instances (the bonus, or the entropy as an output).
bool wants_entropy(const grpo_loss_terms* terms) {
  return terms && (terms->ent_coef != 0.f || terms->entropy_tok != nullptr);
}

int check_args(const void* h, const void* W, int64_t T, int64_t V, int64_t H, const int32_t* target,
               const float* adv_tok, const uint8_t* mask, const float* loss_tok, const grpo_step_acc* acc) {
  if (T < 0 || V < 1 || H < BK || H % BK != 0 || !acc) return GRPO_ERR_INVALID;
  if (T == 0) return GRPO_OK;
  if (!h || !W || !target || !adv_tok || !mask || !loss_tok) return GRPO_ERR_INVALID;
  if (((uintptr_t)h | (uintptr_t)W) & 15u) return GRPO_ERR_INVALID;
  if (T > INT32_MAX / 2 || V > INT32_MAX / 2) return GRPO_ERR_INVALID;
  return GRPO_OK;
}

// Pass A and the per-token reduce: loss_tok, logp_tok, the step counters, and each token's
// LSE and gradient coefficient in the scratch.
int forward(int cg, const void* h, const void* W, int64_t T, int64_t V, int64_t H, const int32_t* target,
            const float* old_logp, const float* adv_tok, const uint8_t* mask, float clip_eps, float grad_scale,
            float* loss_tok, float* logp_tok, const grpo_loss_terms* terms, grpo_step_acc* acc,
            const WsLayout& ws, const Scratch& sc, cudaStream_t st, bool skip_masked = false) {
  const bool ent = wants_entropy(terms);
  GemmArgs g{};
  g.target = target;
  g.part_m = sc.part_m;
  g.part_s = sc.part_s;
  g.part_s2 = sc.part_s2;
  g.zy = sc.zy;
  g.acc = acc;
  g.col_tile0 = 0;
  g.n_n = ws.n_col_tiles;
  const void* a_src = h;
  if (skip_masked) {
    // the valid tokens first (their count on the device) and their hidden states gathered:
    // pass A and the reduce run over those rows only
    partition_kernel<<<1, kPartThreads, 0, st>>>(T, mask, nullptr, nullptr, nullptr, sc.idx, sc.live_n);
    GRPO_CUDA_TRY(cudaGetLastError());
    const int64_t blocks = std::min<int64_t>((T + 7) / 8, (int64_t)sm_count() * 16);
    gather_kernel<<<(unsigned)blocks, 256, 0, st>>>(T, (int)H, static_cast<const __nv_bfloat16*>(h), sc.idx,
                                                    sc.live_n, sc.h_live, nullptr);
    GRPO_CUDA_TRY(cudaGetLastError());
    a_src = sc.h_live;
    g.live_n = sc.live_n;
    g.row_idx = sc.idx;
    g.live_mode = LIVE_ROWS;
  }
  const int rc = ent ? logits_gemm<EPI_PARTIALS_ENT>(cg, a_src, W, T, V, H, g, st)
                     : logits_gemm<EPI_PARTIALS>(cg, a_src, W, T, V, H, g, st);
  if (rc != GRPO_OK) return rc;
  ReduceArgs r{};
  r.T = T;
  r.V = V;
  r.n_col_tiles = ws.n_col_tiles;
  r.part_m = sc.part_m;
  r.part_s = sc.part_s;
  r.part_s2 = sc.part_s2;
  r.zy = sc.zy;
  r.target = target;
  r.old_logp = old_logp;
  r.adv = adv_tok;
  r.mask = mask;
  r.eps = clip_eps;
  r.scale = grad_scale;
  if (terms) {
    r.kl_kind = terms->kl_kind;
    r.kl_coef = terms->kl_coef;
    r.ent_coef = terms->ent_coef;
    r.ref_logp = terms->ref_logp;
    r.w_tok = terms->w_tok;
    r.entropy_tok = terms->entropy_tok;
  }
  r.lse2_out = sc.lse2;
  r.coef_out = sc.coef;
  r.ea_out = sc.ea;
  r.eb_out = sc.eb;
  r.loss_tok = loss_tok;
  r.logp_tok = logp_tok;
  r.acc = acc;
  if (skip_masked) {
    r.idx = sc.idx;
    r.live_n = sc.live_n;
  }
  const dim3 grid((unsigned)((T + 31) / 32)), block(kReduceWarps * 32);
  if (ent)
    reduce_kernel<true, true><<<grid, block, 0, st>>>(r);
  else if (terms)
    reduce_kernel<false, true><<<grid, block, 0, st>>>(r);
  else
    reduce_kernel<false, false><<<grid, block, 0, st>>>(r);
  GRPO_CUDA_TRY(cudaGetLastError());
  return GRPO_OK;
}

// The backward's second stream and its events, one set per device, created by the first call
// that needs them (with the device current) and kept for the process lifetime. A call holds
// `lock` while it enqueues its backward, so calls from several host threads never interleave
// their records of these events; their work on the shared stream runs in enqueue order.
struct Overlap {
  cudaStream_t aux = nullptr;
  cudaEvent_t dz_ready = nullptr, joined = nullptr, buf_free[2] = {nullptr, nullptr};
};

// Whether the next chunk's recompute may run beside this chunk's d_h and dW
// (GRPO_LMHEAD_OVERLAP=0 keeps every launch on the caller's stream).
bool overlap_on() {
  const char* e = getenv("GRPO_LMHEAD_OVERLAP");
  return !(e && e[0] == '0');
}

Overlap* overlap_state(std::unique_lock<std::mutex>& lock) {
  static Overlap per_dev[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return nullptr;
  }
  lock = std::unique_lock<std::mutex>(mu);
  Overlap& o = per_dev[dev];
  if (!o.aux) {
    Overlap n;
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&n.aux, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&n.dz_ready, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&n.joined, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&n.buf_free[0], ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&n.buf_free[1], ef) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;  // (what was created is kept until exit; the call falls back to one stream)
    }
    o = n;
  }
  return &o;
}

}  // namespace

extern "C" GRPO_API size_t grpo_lmhead_workspace_size(int64_t T, int64_t V, int64_t H) {
  if (T <= 0 || V <= 0 || H <= 0) return 0;
  return ws_layout(T, V, H).total;
}

extern "C" GRPO_API int grpo_lmhead_loss_fwd_bwd_ex(const void* h, const void* W, int64_t T, int64_t V,
                                                    int64_t H, const int32_t* target, const float* old_logp,
                                                    const float* adv_tok, const uint8_t* mask, float clip_eps,
                                                    float grad_scale, float* d_h, float* dW, uint32_t flags,
                                                    float* loss_tok, float* logp_tok,
                                                    const grpo_loss_terms* terms, grpo_step_acc* acc,
                                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (terms) {
    if (terms->kl_kind != GRPO_KL_NONE && terms->kl_kind != GRPO_KL_K1 && terms->kl_kind != GRPO_KL_K3)
      return GRPO_ERR_INVALID;
    if (terms->kl_kind != GRPO_KL_NONE && !terms->ref_logp) return GRPO_ERR_INVALID;
    if (!isfinite(terms->kl_coef) || !isfinite(terms->ent_coef)) return GRPO_ERR_INVALID;
  }
  const int arc = check_args(h, W, T, V, H, target, adv_tok, mask, loss_tok, acc);
  if (arc != GRPO_OK || T == 0) return arc;
  if (flags & ~(uint32_t)(GRPO_LMHEAD_DW_ACCUMULATE | GRPO_LMHEAD_SKIP_MASKED)) return GRPO_ERR_INVALID;
  if (!workspace || ((uintptr_t)workspace & 255u)) return GRPO_ERR_INVALID;
  if (((uintptr_t)d_h | (uintptr_t)dW) & 15u) return GRPO_ERR_INVALID;  // 16-byte row stores
  const WsLayout ws = ws_layout(T, V, H);
  if (workspace_bytes < ws.total) return GRPO_ERR_CAPACITY;
  const cudaStream_t st = as_stream(stream);
  const Scratch sc = carve(workspace, ws, true);
  const int cg = cta_group();
  int rc = forward(cg, h, W, T, V, H, target, old_logp, adv_tok, mask, clip_eps, grad_scale, loss_tok, logp_tok,
                   terms, acc, ws, sc, st, (flags & GRPO_LMHEAD_SKIP_MASKED) != 0);
  if (rc != GRPO_OK || (!d_h && !dW)) return rc;
  // the dlogits take the entropy form p (ea + eb z) when the bonus has a coefficient
  const bool ent_grad = terms && terms->ent_coef != 0.f;

  // Per vocabulary chunk c: the recompute writes the chunk's dlogits into buffer c % 2 on the
  // caller's stream; d_h and dW read it on the second stream, so the next chunk's recompute
  // runs beside them. d_h's launches stay in chunk order on one stream (its accumulation
  // order), and a buffer is rewritten only after the launches reading it two chunks before.
  const int n_chunks = (ws.n_col_tiles + ws.chunk_tiles - 1) / ws.chunk_tiles;
  std::unique_lock<std::mutex> ov_lock;
  Overlap* ov = (overlap_on() && n_chunks > 1) ? overlap_state(ov_lock) : nullptr;
  const cudaStream_t bst = ov ? ov->aux : st;  // the stream of d_h and dW
  const __nv_bfloat16* Wb = static_cast<const __nv_bfloat16*>(W);
  // the live tokens in a compact order, their hidden states gathered; the dead tokens' d_h rows
  // zeroed
  partition_kernel<<<1, kPartThreads, 0, st>>>(T, nullptr, sc.coef, ent_grad ? sc.ea : nullptr,
                                                ent_grad ? sc.eb : nullptr, sc.idx, sc.live_n);
  GRPO_CUDA_TRY(cudaGetLastError());
  {
    const int64_t blocks = std::min<int64_t>((T + 7) / 8, (int64_t)sm_count() * 16);
    gather_kernel<<<(unsigned)blocks, 256, 0, st>>>(T, (int)H, static_cast<const __nv_bfloat16*>(h), sc.idx, sc.live_n,
                                                    sc.h_live, d_h);
    GRPO_CUDA_TRY(cudaGetLastError());
  }
  auto backward = [&]() -> int {
  for (int ct0 = 0, c = 0; ct0 < ws.n_col_tiles; ct0 += ws.chunk_tiles, ++c) {
    const int nct = std::min(ws.chunk_tiles, ws.n_col_tiles - ct0);
    const int64_t v0 = (int64_t)ct0 * BN;
    const int64_t vc = std::min<int64_t>((int64_t)nct * BN, V - v0);
    __nv_bfloat16* dzb = sc.dz[ov ? (c & 1) : 0];
    if (ov && c >= 2) GRPO_CUDA_TRY(cudaStreamWaitEvent(st, ov->buf_free[c & 1], 0));
    // the chunk's dlogits, recomputed from its logits
    GemmArgs g{};
    g.target = target;
    g.lse2 = sc.lse2;
    g.coef = sc.coef;
    if (ent_grad) {
      g.ea = sc.ea;
      g.eb = sc.eb;
    }
    g.dz = dzb;
    g.ldz = ws.vchunk;
    g.v0 = v0;
    g.acc = acc;
    g.col_tile0 = ct0;
    g.n_n = nct;
    g.live_n = sc.live_n;  // compact rows; zero dlogits rows up to the padded live count
    g.row_idx = sc.idx;
    g.live_mode = LIVE_ROWS_PADDED;
    rc = logits_gemm<EPI_DLOGITS>(cg, sc.h_live, W, T, V, H, g, st, vc);
    if (rc != GRPO_OK) return rc;
    if (ov) {
      GRPO_CUDA_TRY(cudaEventRecord(ov->dz_ready, st));
      GRPO_CUDA_TRY(cudaStreamWaitEvent(bst, ov->dz_ready, 0));
    }
    CUtensorMap ma, mb;
    if (d_h) {
      // d_h[live rows, H] (+)= dz_c[live rows, vc] W_c[vc, H], each row stored to its token's row
      if (!map_k(&ma, dzb, T, vc, ws.vchunk, BM) || !map_mn(&mb, Wb + v0 * H, vc, H, H))
        return GRPO_ERR_UNSUPPORTED;
      GemmArgs b{};
      b.live_n = sc.live_n;
      b.row_idx = sc.idx;
      b.live_mode = LIVE_ROWS;
      b.M = T;
      b.N = H;
      b.K = vc;
      b.n_n = (int)((H + BN - 1) / BN);
      b.m_fast = 0;  // consecutive units share the dz rows
      b.C = d_h;
      b.ldc = H;
      b.accumulate = c > 0;
      b.acc = acc;
      rc = launch<EPI_STORE_F32, false, true>(cg, ma, mb, ma, b, bst);
      if (rc != GRPO_OK) return rc;
    }
    if (dW) {
      // dW_c[vc, H] = dz_c^T[vc, live] h_live[live, H], reduced over the padded live count
      if (!map_mn(&ma, dzb, T, vc, ws.vchunk) || !map_mn(&mb, sc.h_live, T, H, H)) return GRPO_ERR_UNSUPPORTED;
      GemmArgs b{};
      b.live_n = sc.live_n;
      b.live_mode = LIVE_K;
      b.M = vc;
      b.N = H;
      b.K = T;
      b.n_n = (int)((H + BN - 1) / BN);
      b.m_fast = 0;  // consecutive units share the dz columns
      b.C = dW + v0 * H;
      b.ldc = H;
      b.accumulate = (flags & GRPO_LMHEAD_DW_ACCUMULATE) ? 1 : 0;
      b.acc = acc;
      rc = launch<EPI_STORE_F32, true, true>(cg, ma, mb, ma, b, bst);
      if (rc != GRPO_OK) return rc;
    }
    if (ov) GRPO_CUDA_TRY(cudaEventRecord(ov->buf_free[c & 1], bst));
  }
  return GRPO_OK;
  };
  rc = backward();
  if (ov) {  // the caller's stream continues after every launch of the call (also after an error)
    const bool joined = cudaEventRecord(ov->joined, bst) == cudaSuccess &&
                        cudaStreamWaitEvent(st, ov->joined, 0) == cudaSuccess;
    if (!joined) {
      (void)cudaGetLastError();
      if (rc == GRPO_OK) rc = GRPO_ERR_CUDA;
    }
  }
  return rc;
}

extern "C" GRPO_API int grpo_lmhead_loss_fwd_bwd(const void* h, const void* W, int64_t T, int64_t V, int64_t H,
                                                 const int32_t* target, const float* old_logp,
                                                 const float* adv_tok, const uint8_t* mask, float clip_eps,
                                                 float grad_scale, float* d_h, float* dW, uint32_t flags,
                                                 float* loss_tok, float* logp_tok, grpo_step_acc* acc,
                                                 void* workspace, size_t workspace_bytes, void* stream) {
  return grpo_lmhead_loss_fwd_bwd_ex(h, W, T, V, H, target, old_logp, adv_tok, mask, clip_eps, grad_scale, d_h, dW,
                                     flags, loss_tok, logp_tok, nullptr, acc, workspace, workspace_bytes, stream);
}

// ---- allocation-free forward entry point -----------------------------------------------------
//
// For callers that cannot allocate device memory when they need the loss: a serving or
// scoring process that has handed all device memory to its own pool (KV cache, a caching
// allocator) so that a fresh cudaMalloc would fail or force the pool to shrink, or a code path
// that must not risk the implicit device synchronisation that cudaMalloc / cudaFree can
// cause. Such a caller still passes its inputs and outputs; the forward pass's scratch
// (per-token vocabulary-tile softmax partials, target logits, LSE, coefficients) lives in the
// file-scope array below instead of a caller workspace.
//
// The array is a device symbol: every GPU that loads this library holds its 16 MiB until the
// process exits. In host code its name only stands in for the symbol; its device address is
// looked up by cudaGetSymbolAddress (with the device current) and passed to the kernels.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
static __device__ __align__(256) unsigned char g_lmhead_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Unique id of the calling thread's current context (cuCtxGetId), or 0 if unavailable.
unsigned long long current_ctx_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch array in the current device's context. The first call on a
// device (and the first after that device's primary context was destroyed and re-created, e.g.
// by cudaDeviceReset: the context id changes) looks it up and records it with the context id;
// later calls in the same context reuse it without any CUDA call but the id query.
int noalloc_setup(void** scratch) {
  static void* addr[64] = {};
  static unsigned long long ctx_of[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return GRPO_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return GRPO_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long id = addr[dev] ? current_ctx_id() : 0;
  if (!addr[dev] || id == 0 || id != ctx_of[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_lmhead_noalloc_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return GRPO_ERR_CUDA;
    }
    addr[dev] = p;
    ctx_of[dev] = current_ctx_id();
  }
  *scratch = addr[dev];
  return GRPO_OK;
}

}  // namespace

extern "C" GRPO_API size_t grpo_lmhead_forward_noalloc_max_scratch(void) { return kNoAllocScratchBytes; }

extern "C" GRPO_API int grpo_lmhead_forward_noalloc(const void* h, const void* W, int64_t T, int64_t V,
                                                    int64_t H, const int32_t* target, const float* old_logp,
                                                    const float* adv_tok, const uint8_t* mask, float clip_eps,
                                                    float grad_scale, float* loss_tok, float* logp_tok,
                                                    grpo_step_acc* acc, void* stream) {
  const int arc = check_args(h, W, T, V, H, target, adv_tok, mask, loss_tok, acc);
  if (arc != GRPO_OK || T == 0) return arc;
  // the forward pass uses the workspace layout up to (not including) the dlogits chunk
  const WsLayout ws = ws_layout(T, V, H);
  if (ws.dz > kNoAllocScratchBytes) return GRPO_ERR_CAPACITY;
  void* scratch = nullptr;
  const int rc = noalloc_setup(&scratch);
  if (rc != GRPO_OK) return rc;
  return forward(cta_group(), h, W, T, V, H, target, old_logp, adv_tok, mask, clip_eps, grad_scale, loss_tok,
                 logp_tok, nullptr, acc, ws, carve(scratch, ws, false), as_stream(stream));
}
