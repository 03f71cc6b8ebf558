/* A plain-C client of libgrpo's fused LM-head variant, with nothing but grpo.h and the CUDA
 * runtime: one call with d_h and dW (the workspace sized by grpo_lmhead_workspace_size) and the
 * step finish, then a second step through grpo_lmhead_loss_fwd_bwd_ex with the regularisers
 * (KL k3 to ref_logp, the entropy bonus with the entropy written per token) and the
 * GRPO_LMHEAD_SKIP_MASKED flag, and its finish. The parity test writes the inputs, runs this
 * program and compares its outputs with the Python binding's on the same inputs.
 *
 *   lmhead_step <in> <out>
 * in  (little-endian): int64 T, int64 V, int64 H, float clip_eps, float grad_scale,
 *     uint16 h[T*H] (bf16 bits), uint16 W[V*H] (bf16 bits), int32 target[T], float old_logp[T],
 *     float adv[T], uint8 mask[T], float ref_logp[T]
 * out, per step (the plain one, then the regularised one): int32 status of the finish,
 *     float loss_tok[T], float logp_tok[T], float d_h[T*H], float dW[V*H], double loss,
 *     int64 n_valid, int64 n_clipped; then float entropy[T] of the second step */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "grpo.h"

static int read_all(FILE* f, void* p, size_t n) { return fread(p, 1, n, f) == n; }
static int write_all(FILE* f, const void* p, size_t n) { return fwrite(p, 1, n, f) == n; }

#define CK(x)                                              \
  do {                                                     \
    if ((x) != cudaSuccess) {                              \
      fprintf(stderr, "CUDA call failed: %s\n", #x);       \
      return 2;                                            \
    }                                                      \
  } while (0)

/* host buffer -> new device buffer */
static int upload(void** d, const void* h, size_t n) {
  if (cudaMalloc(d, n) != cudaSuccess) return 0;
  return cudaMemcpy(*d, h, n, cudaMemcpyHostToDevice) == cudaSuccess;
}

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: lmhead_step <in> <out>\n");
    return 1;
  }
  FILE* fi = fopen(argv[1], "rb");
  if (!fi) return 1;
  int64_t T = 0, V = 0, H = 0;
  float eps = 0.f, scale = 0.f;
  if (!read_all(fi, &T, 8) || !read_all(fi, &V, 8) || !read_all(fi, &H, 8) || !read_all(fi, &eps, 4) ||
      !read_all(fi, &scale, 4))
    return 1;
  const size_t nh = (size_t)T * (size_t)H, nw = (size_t)V * (size_t)H;
  uint16_t* h = malloc(nh * 2);
  uint16_t* w = malloc(nw * 2);
  int32_t* tgt = malloc((size_t)T * 4);
  float* old = malloc((size_t)T * 4);
  float* adv = malloc((size_t)T * 4);
  uint8_t* mask = malloc((size_t)T);
  float* loss = malloc((size_t)T * 4);
  float* logp = malloc((size_t)T * 4);
  float* dh = malloc(nh * 4);
  float* dw = malloc(nw * 4);
  float* ref = malloc((size_t)T * 4);
  float* ent = malloc((size_t)T * 4);
  if (!h || !w || !tgt || !old || !adv || !mask || !loss || !logp || !dh || !dw || !ref || !ent) return 1;
  if (!read_all(fi, h, nh * 2) || !read_all(fi, w, nw * 2) || !read_all(fi, tgt, (size_t)T * 4) ||
      !read_all(fi, old, (size_t)T * 4) || !read_all(fi, adv, (size_t)T * 4) || !read_all(fi, mask, (size_t)T) ||
      !read_all(fi, ref, (size_t)T * 4))
    return 1;
  fclose(fi);

  void *d_h, *d_w, *d_tgt, *d_old, *d_adv, *d_mask, *d_loss, *d_logp, *d_dh, *d_dw, *d_acc, *d_ws, *d_ref, *d_ent;
  if (!upload(&d_h, h, nh * 2) || !upload(&d_w, w, nw * 2) || !upload(&d_tgt, tgt, (size_t)T * 4) ||
      !upload(&d_old, old, (size_t)T * 4) || !upload(&d_adv, adv, (size_t)T * 4) ||
      !upload(&d_mask, mask, (size_t)T) || !upload(&d_ref, ref, (size_t)T * 4))
    return 2;
  CK(cudaMalloc(&d_ent, (size_t)T * 4));
  const size_t ws_bytes = grpo_lmhead_workspace_size(T, V, H);
  if (ws_bytes == 0) return 1;
  CK(cudaMalloc(&d_loss, (size_t)T * 4));
  CK(cudaMalloc(&d_logp, (size_t)T * 4));
  CK(cudaMalloc(&d_dh, nh * 4));
  CK(cudaMalloc(&d_dw, nw * 4));
  CK(cudaMalloc(&d_ws, ws_bytes)); /* cudaMalloc returns 256-byte aligned memory */
  CK(cudaMalloc(&d_acc, sizeof(grpo_step_acc)));
  CK(cudaMemset(d_acc, 0, sizeof(grpo_step_acc)));

  FILE* fo = fopen(argv[2], "wb");
  if (!fo) return 1;
  for (int pass = 0; pass < 2; ++pass) {
    CK(cudaMemset(d_acc, 0, sizeof(grpo_step_acc)));
    int rc;
    if (pass == 0) {
      rc = grpo_lmhead_loss_fwd_bwd(d_h, d_w, T, V, H, d_tgt, d_old, d_adv, d_mask, eps, scale, d_dh, d_dw, 0u,
                                    d_loss, d_logp, d_acc, d_ws, ws_bytes, NULL);
    } else {
      grpo_loss_terms terms = {GRPO_KL_K3, 0.1f, (const float*)d_ref, 0.02f, (float*)d_ent, NULL};
      rc = grpo_lmhead_loss_fwd_bwd_ex(d_h, d_w, T, V, H, d_tgt, d_old, d_adv, d_mask, eps, scale, d_dh, d_dw,
                                       GRPO_LMHEAD_SKIP_MASKED, d_loss, d_logp, &terms, d_acc, d_ws, ws_bytes,
                                       NULL);
    }
    if (rc != GRPO_OK) {
      fprintf(stderr, "grpo_lmhead_loss_fwd_bwd (step %d): %s\n", pass, grpo_status_string(rc));
      return 3;
    }
    grpo_step_result res;
    const int st = grpo_finish_step(d_acc, d_loss, T, -1, 0, NULL, NULL, NULL, 0, &res, NULL);
    if (st < 0 && st != GRPO_ERR_N_MISMATCH) {
      fprintf(stderr, "grpo_finish_step: %s\n", grpo_status_string(st));
      return 3;
    }
    CK(cudaMemcpy(loss, d_loss, (size_t)T * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(logp, d_logp, (size_t)T * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(dh, d_dh, nh * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(dw, d_dw, nw * 4, cudaMemcpyDeviceToHost));
    const int32_t st32 = st;
    if (!write_all(fo, &st32, 4) || !write_all(fo, loss, (size_t)T * 4) || !write_all(fo, logp, (size_t)T * 4) ||
        !write_all(fo, dh, nh * 4) || !write_all(fo, dw, nw * 4) || !write_all(fo, &res.loss, 8) ||
        !write_all(fo, &res.n_valid, 8) || !write_all(fo, &res.n_clipped, 8))
      return 1;
  }
  CK(cudaMemcpy(ent, d_ent, (size_t)T * 4, cudaMemcpyDeviceToHost));
  if (!write_all(fo, ent, (size_t)T * 4)) return 1;
  fclose(fo);
  void* bufs[] = {d_h, d_w, d_tgt, d_old, d_adv, d_mask, d_loss, d_logp, d_dh, d_dw, d_ws, d_acc, d_ref, d_ent};
  for (size_t i = 0; i < sizeof(bufs) / sizeof(bufs[0]); ++i) cudaFree(bufs[i]);
  free(h); free(w); free(tgt); free(old); free(adv); free(mask); free(loss); free(logp); free(dh); free(dw);
  free(ref); free(ent);
  return 0;
}
