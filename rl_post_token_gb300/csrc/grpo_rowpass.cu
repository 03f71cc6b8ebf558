// Row pass: launch configuration, kernel selection and the C entry points. The kernels and
// the layout of their arguments are in grpo_rowpass_kernels.cuh.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "grpo_rowpass_kernels.cuh"

namespace grpo {

size_t max_smem_optin();

// Launches a persistent cluster kernel with as many clusters as fit on the device at once
// (no more than there are rows). Per device and kernel: the kernel's shared-memory limit only
// ever rises (a concurrent launch with a larger slice never finds it lowered under it), and
// the co-resident cluster count is cached per shared-memory size.
template <auto KERN>
int launch_clusters(const RowArgs& a, int C, int threads, size_t smem, int Vs, int S, cudaStream_t st) {
  int dev = 0;
  GRPO_CUDA_TRY(cudaGetDevice(&dev));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n_clusters = 0;
  {
    struct Entry { size_t smem; int clusters; };
    static std::mutex mu;
    static size_t limit[64] = {};
    static Entry seen[64][4] = {};
    std::lock_guard<std::mutex> lock(mu);
    const bool known_dev = dev >= 0 && dev < 64;
    if (known_dev)
      for (const Entry& e : seen[dev])
        if (e.smem == smem) n_clusters = e.clusters;
    if (n_clusters == 0) {
      if (!known_dev || smem > limit[dev]) {
        GRPO_CUDA_TRY(cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        if (known_dev) limit[dev] = smem;
      }
      cfg.gridDim = dim3(C * 1024, 1, 1);
      GRPO_CUDA_TRY(cudaOccupancyMaxActiveClusters(&n_clusters, KERN, &cfg));
      if (n_clusters < 1) return GRPO_ERR_UNSUPPORTED;
      if (known_dev) {
        Entry* slot = &seen[dev][0];
        for (Entry& e : seen[dev])
          if (e.smem == 0) { slot = &e; break; }
        *slot = Entry{smem, n_clusters};
      }
    }
  }
  const int64_t clusters = std::min<int64_t>(a.T, n_clusters);
  cfg.gridDim = dim3((unsigned)(clusters * C), 1, 1);
  GRPO_CUDA_TRY(cudaLaunchKernelEx(&cfg, KERN, a, Vs, S));
  return GRPO_OK;
}

template <typename T, int C, int NCW, int VPT, int MINB, bool ENT, int TERMS>
int launch_cluster(const RowArgs& a, cudaStream_t st) {
  constexpr int CH = cluster_chunk_elems<T>(NCW, VPT);
  const int Vs = cluster_slice_elems<T>(a.V, C);
  const int nchm = (Vs + CH - 1) / CH;
  if (nchm > kMaxChunks) return GRPO_ERR_UNSUPPORTED;
  // Ring slots: a CTA alone on its SM takes as many chunk slots as the opt-in shared memory
  // holds (the spare ones carry the next row); CTAs that share an SM keep the fixed buffer.
  int S = nchm;
  int s_fit = 0;
  const size_t optin = max_smem_optin();
  if (MINB == 1 && optin > cluster_tail_bytes(NCW)) {
    s_fit = (int)std::min<size_t>(kMaxChunks, (optin - cluster_tail_bytes(NCW)) / ((size_t)CH * sizeof(T)));
    if (s_fit > nchm) S = s_fit;
  }
  if (const char* ov = getenv("GRPO_ROWPASS_SLOTS")) {  // 0: fixed buffer; n: n slots if they fit
    const int n = atoi(ov);
    if (n == 0) S = nchm;
    else if (n > nchm && n <= s_fit) S = n;
  }
  const size_t smem = cluster_ring_bytes<T>(Vs, CH, S) + cluster_tail_bytes(NCW);
  return launch_clusters<row_cluster_kernel<T, C, NCW, VPT, MINB, ENT, TERMS>>(a, C, (NCW + 1) * 32, smem, Vs, S,
                                                                               st);
}

// The forward-only streaming kernel: as many ring slots as the opt-in shared memory holds (at
// least 2; GRPO_ROWPASS_SLOTS=n takes n of them, 0 the minimum), whatever the row length.
template <typename T, int C, int NCW, int VPT>
int launch_fwd(const RowArgs& a, cudaStream_t st) {
  constexpr int CH = cluster_chunk_elems<T>(NCW, VPT);
  const int Vs = cluster_slice_elems<T>(a.V, C);
  const size_t optin = max_smem_optin();
  const size_t tail = fwd_tail_bytes(C, NCW);
  if (optin <= tail) return GRPO_ERR_UNSUPPORTED;
  const int s_fit = (int)std::min<size_t>(kMaxChunks, (optin - tail) / ((size_t)CH * sizeof(T)));
  if (s_fit < 2) return GRPO_ERR_UNSUPPORTED;
  int S = s_fit;
  if (const char* ov = getenv("GRPO_ROWPASS_SLOTS")) {
    const int n = atoi(ov);
    S = n < 2 ? 2 : std::min(n, s_fit);
  }
  const size_t smem = (size_t)S * CH * sizeof(T) + tail;
  return launch_clusters<row_fwd_kernel<T, C, NCW, VPT>>(a, C, fwd_block_threads(NCW), smem, Vs, S, st);
}

template <typename T, int NT, int U, bool ENT, int TERMS>
int launch_l2(const RowArgs& a, bool vec, int blocks_per_sm, cudaStream_t st) {
  const int64_t grid = std::min<int64_t>(a.T, (int64_t)sm_count() * blocks_per_sm);
  if (vec)
    row_l2_kernel<T, NT, U, true, ENT, TERMS><<<(unsigned)grid, NT, 0, st>>>(a);
  else
    row_l2_kernel<T, NT, U, false, ENT, TERMS><<<(unsigned)grid, NT, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? GRPO_OK : GRPO_ERR_CUDA;
}

size_t max_smem_optin() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cached[dev].load(std::memory_order_relaxed) > 0) return (size_t)cached[dev].load();
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || n < 0) n = 0;
  if (dev >= 0 && dev < 64) cached[dev].store(n);
  return (size_t)n;
}

int sm_count() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cached[dev].load(std::memory_order_relaxed) > 0) return cached[dev].load();
  int n = 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  if (dev >= 0 && dev < 64) cached[dev].store(n);
  return n;
}

}  // namespace grpo

using namespace grpo;

namespace {

// Whether the cluster kernel fits: the fixed staging buffer of `minb` CTAs in the shared memory
// of one SM, and the slice in at most kMaxChunks chunks.
template <typename T>
bool cluster_fits(int64_t V, int C, int NCW, int minb, int vpt) {
  const int64_t cap = 227 * 1024;
  const int Vs = cluster_slice_elems<T>(V, C);
  return (int64_t)cluster_smem_bytes<T>(Vs, NCW) * minb <= cap &&
         (Vs + cluster_chunk_elems<T>(NCW, vpt) - 1) / cluster_chunk_elems<T>(NCW, vpt) <= kMaxChunks;
}

// Forward-only calls without extra terms take the streaming kernel unless GRPO_ROWPASS_FWD=0
// (the general cluster kernel, which gives the same bits).
bool fwd_kernel_on() {
  const char* v = getenv("GRPO_ROWPASS_FWD");
  return !(v && strcmp(v, "0") == 0);
}

template <bool ENT, int TERMS>
int dispatch(const RowArgs& a, int32_t dtype, bool vec, cudaStream_t st) {
  const int64_t V = a.V;
  const char* pin = getenv("GRPO_ROWPASS");
  const bool pin_l2 = pin && strcmp(pin, "l2") == 0;
  // every instance runs 32 KB chunks where one CTA has an SM to itself; where two CTAs share
  // an SM (c3/c4) the entropy instances take half-size chunks to stay in registers
  if (dtype == GRPO_DTYPE_BF16) {
    // Large bf16 vocabularies: rows split across a CTA cluster, slices staged in shared
    // memory. Variants (cluster size, consumer warps, vectors per thread, CTAs per SM):
    // c2 = (2, 16, 4, 1) with a ring of spare slots, c3 = (3, 8, 4, 2), c4 = (4, 8, 4, 2)
    // with fixed staging buffers.
    using B16 = __nv_bfloat16;
    if (vec && V % 8 == 0 && V >= 16384 && !pin_l2) {
      auto c34 = [&](auto c_tag) {
        constexpr int C = decltype(c_tag)::value;
        if constexpr (ENT)
          if (cluster_fits<B16>(V, C, 8, 2, 2)) return launch_cluster<B16, C, 8, 2, 2, ENT, TERMS>(a, st);
        return launch_cluster<B16, C, 8, 4, 2, ENT, TERMS>(a, st);
      };
      using C3 = std::integral_constant<int, 3>;
      using C4 = std::integral_constant<int, 4>;
      if (pin && strcmp(pin, "c3") == 0 && cluster_fits<B16>(V, 3, 8, 2, 4)) return c34(C3{});
      if (pin && strcmp(pin, "c4") == 0 && cluster_fits<B16>(V, 4, 8, 2, 4)) return c34(C4{});
      if (cluster_fits<B16>(V, 2, 16, 1, 4)) {
        if constexpr (!ENT && TERMS == 0)
          if (!a.dlogits && fwd_kernel_on()) return launch_fwd<B16, 2, 16, 4>(a, st);
        return launch_cluster<B16, 2, 16, 4, 1, ENT, TERMS>(a, st);
      }
      if (cluster_fits<B16>(V, 4, 8, 2, 4)) return c34(C4{});
      if (cluster_fits<B16>(V, 4, 16, 1, 4)) {
        if constexpr (!ENT && TERMS == 0)
          if (!a.dlogits && fwd_kernel_on()) return launch_fwd<B16, 4, 16, 4>(a, st);
        return launch_cluster<B16, 4, 16, 4, 1, ENT, TERMS>(a, st);
      }
    }
    if (V >= 8192) return launch_l2<B16, 1024, 2, ENT, TERMS>(a, vec, 1, st);
    return launch_l2<B16, 128, 2, ENT, TERMS>(a, vec, 16, st);
  }
  // float32 vocabularies: a row is twice the bytes, so a 4-CTA cluster, one CTA per SM with
  // the ring of spare slots, holds the same slice size as the bf16 2-CTA cluster
  if (vec && V % 4 == 0 && V >= 16384 && !pin_l2 && cluster_fits<float>(V, 4, 16, 1, 4)) {
    if constexpr (!ENT && TERMS == 0)
      if (!a.dlogits && fwd_kernel_on()) return launch_fwd<float, 4, 16, 4>(a, st);
    return launch_cluster<float, 4, 16, 4, 1, ENT, TERMS>(a, st);
  }
  if (V >= 8192) return launch_l2<float, 1024, 2, ENT, TERMS>(a, vec, 1, st);
  return launch_l2<float, 128, 2, ENT, TERMS>(a, vec, 16, st);
}

}  // namespace

extern "C" GRPO_API int grpo_logprob_loss_fwd_bwd_ex(const void* logits, int32_t dtype, int64_t T, int64_t V,
                                                     int64_t ld, const int64_t* tok_src, const int32_t* target,
                                                     const float* old_logp, const float* adv_tok,
                                                     const uint8_t* mask, float clip_eps, float grad_scale,
                                                     void* dlogits, int64_t ld_out, float* loss_tok,
                                                     float* logp_tok, const grpo_loss_terms* terms,
                                                     grpo_step_acc* acc, void* stream) {
  if (dtype != GRPO_DTYPE_F32 && dtype != GRPO_DTYPE_BF16) return GRPO_ERR_UNSUPPORTED;
  if (T < 0 || V < 1 || ld < V || !acc) return GRPO_ERR_INVALID;
  if (dlogits && ld_out < V) return GRPO_ERR_INVALID;
  if (terms) {
    if (terms->kl_kind != GRPO_KL_NONE && terms->kl_kind != GRPO_KL_K1 && terms->kl_kind != GRPO_KL_K3)
      return GRPO_ERR_INVALID;
    if (terms->kl_kind != GRPO_KL_NONE && !terms->ref_logp) return GRPO_ERR_INVALID;
    if (!isfinite(terms->kl_coef) || !isfinite(terms->ent_coef)) return GRPO_ERR_INVALID;
  }
  if (T == 0) return GRPO_OK;
  if (!logits || !target || !adv_tok || !mask || !loss_tok) return GRPO_ERR_INVALID;
  if (V > (int64_t)INT32_MAX || T > (int64_t)INT32_MAX) return GRPO_ERR_INVALID;

  RowArgs a{logits, T, V, ld, tok_src, target, old_logp, adv_tok, mask, clip_eps, grad_scale,
            dlogits, ld_out, loss_tok, logp_tok, acc,
            terms ? terms->kl_kind : 0, terms ? terms->kl_coef : 0.f,
            terms && terms->kl_kind ? terms->ref_logp : nullptr, terms ? terms->ent_coef : 0.f,
            terms ? terms->entropy_tok : nullptr, terms ? terms->w_tok : nullptr};
  const cudaStream_t st = as_stream(stream);
  const size_t es = dtype == GRPO_DTYPE_F32 ? 4 : 2;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const bool vec = al16(logits) && (ld * es) % 16 == 0 &&
                   (!dlogits || (al16(dlogits) && (ld_out * es) % 16 == 0));
  // Kernel instances by the work a call needs: the entropy (as a loss term or as an output)
  // needs sum_v p_v z_v, a third accumulator; the KL term a reference log-prob per row; the
  // aggregation weights a weight per row. Each instance carries only its own state, so none
  // pays for the others' registers.
  constexpr int R = kTermsReg, W = kTermsWeight;
  const bool wt = terms && terms->w_tok;
  const bool ent = terms && (terms->ent_coef != 0.f || terms->entropy_tok);
  const bool kl = terms && terms->kl_kind != GRPO_KL_NONE;
  if (ent) return wt ? dispatch<true, R | W>(a, dtype, vec, st) : dispatch<true, R>(a, dtype, vec, st);
  if (kl) return wt ? dispatch<false, R | W>(a, dtype, vec, st) : dispatch<false, R>(a, dtype, vec, st);
  if (wt) return dispatch<false, W>(a, dtype, vec, st);
  return dispatch<false, 0>(a, dtype, vec, st);
}

extern "C" GRPO_API int grpo_logprob_loss_fwd_bwd(const void* logits, int32_t dtype, int64_t T, int64_t V,
                                                  int64_t ld, const int64_t* tok_src, const int32_t* target,
                                                  const float* old_logp, const float* adv_tok,
                                                  const uint8_t* mask, float clip_eps, float grad_scale,
                                                  void* dlogits, int64_t ld_out, float* loss_tok,
                                                  float* logp_tok, grpo_step_acc* acc, void* stream) {
  return grpo_logprob_loss_fwd_bwd_ex(logits, dtype, T, V, ld, tok_src, target, old_logp, adv_tok, mask,
                                      clip_eps, grad_scale, dlogits, ld_out, loss_tok, logp_tok, nullptr, acc,
                                      stream);
}

namespace {

// The events of one host-input call, destroyed when it returns (a pending event may be
// destroyed: its resources go once it completes).
struct CallEvents {
  cudaEvent_t ev[5] = {};
  int n = 0;
  bool create() {
    for (; n < 5; ++n)
      if (cudaEventCreateWithFlags(&ev[n], cudaEventDisableTiming) != cudaSuccess) return false;
    return true;
  }
  ~CallEvents() {
    for (int i = 0; i < n; ++i) cudaEventDestroy(ev[i]);
  }
};

}  // namespace

extern "C" GRPO_API int grpo_logprob_loss_fwd_bwd_host(const void* logits_host, int32_t dtype, int64_t T, int64_t V,
                                                       int64_t ld, const int64_t* tok_src, const int32_t* target,
                                                       const float* old_logp, const float* adv_tok,
                                                       const uint8_t* mask, float clip_eps, float grad_scale,
                                                       void* dlogits, int64_t ld_out, float* loss_tok,
                                                       float* logp_tok, const grpo_loss_terms* terms,
                                                       grpo_step_acc* acc, void* staging, int64_t block_rows,
                                                       void* stream, void* copy_stream) {
  if (dtype != GRPO_DTYPE_F32 && dtype != GRPO_DTYPE_BF16) return GRPO_ERR_UNSUPPORTED;
  if (T < 0 || V < 1 || ld < V || !acc || block_rows < 1) return GRPO_ERR_INVALID;
  if (dlogits && ld_out < V) return GRPO_ERR_INVALID;
  if (T == 0) return GRPO_OK;
  if (!logits_host || !staging || (reinterpret_cast<uintptr_t>(staging) & 15u)) return GRPO_ERR_INVALID;
  if (!target || !adv_tok || !mask || !loss_tok) return GRPO_ERR_INVALID;
  const size_t es = dtype == GRPO_DTYPE_F32 ? 4 : 2;
  const int64_t br = std::min(block_rows, T);
  const size_t row_bytes = (size_t)ld * es;
  const size_t half = (size_t)br * row_bytes;
  const cudaStream_t st = as_stream(stream), cs = as_stream(copy_stream);
  CallEvents e;  // ev[0..1]: block copied into half b; ev[2..3]: half b read; ev[4]: call start
  if (!e.create()) return GRPO_ERR_CUDA;
  // the first copies wait for what is already on `stream` (an earlier call may still read
  // the staging buffer)
  GRPO_CUDA_TRY(cudaEventRecord(e.ev[4], st));
  GRPO_CUDA_TRY(cudaStreamWaitEvent(cs, e.ev[4], 0));
  const bool perm = tok_src != nullptr;
  const uint8_t* src = static_cast<const uint8_t*>(logits_host);
  for (int64_t r0 = 0, k = 0; r0 < T; r0 += br, ++k) {
    const int64_t n = std::min(br, T - r0);
    const int b = (int)(k & 1);
    uint8_t* dst = static_cast<uint8_t*>(staging) + (size_t)b * half;
    if (k >= 2) GRPO_CUDA_TRY(cudaStreamWaitEvent(cs, e.ev[2 + b], 0));  // block k-2's row pass is done
    GRPO_CUDA_TRY(cudaMemcpyAsync(dst, src + (size_t)r0 * row_bytes, (size_t)n * row_bytes,
                                  cudaMemcpyHostToDevice, cs));
    GRPO_CUDA_TRY(cudaEventRecord(e.ev[b], cs));
    GRPO_CUDA_TRY(cudaStreamWaitEvent(st, e.ev[b], 0));
    // the block's rows: side arrays and outputs follow the rows unless read through tok_src
    grpo_loss_terms tb;
    const grpo_loss_terms* tp = nullptr;
    if (terms) {
      tb = *terms;
      if (!perm) {
        if (tb.ref_logp) tb.ref_logp += r0;
        if (tb.entropy_tok) tb.entropy_tok += r0;
        if (tb.w_tok) tb.w_tok += r0;
      }
      tp = &tb;
    }
    const int64_t o = perm ? 0 : r0;
    const int rc = grpo_logprob_loss_fwd_bwd_ex(
        dst, dtype, n, V, ld, perm ? tok_src + r0 : nullptr, target + o, old_logp ? old_logp + o : nullptr,
        adv_tok + o, mask + o, clip_eps, grad_scale,
        dlogits ? static_cast<uint8_t*>(dlogits) + (size_t)r0 * (size_t)ld_out * es : nullptr, ld_out, loss_tok + o,
        logp_tok ? logp_tok + o : nullptr, tp, acc, stream);
    if (rc != GRPO_OK) return rc;
    GRPO_CUDA_TRY(cudaEventRecord(e.ev[2 + b], st));
  }
  return GRPO_OK;
}
