/* A plain-C client of libgrpo: one row pass (log-softmax, clipped surrogate, dlogits) and the
 * step finish over inputs read from a file, with nothing but grpo.h and the CUDA runtime.
 * The parity test writes the inputs, runs this program and compares its outputs with the
 * Python binding's on the same inputs.
 *
 *   loss_step <in> <out>
 * in  (little-endian): int64 T, int64 V, float clip_eps, float grad_scale,
 *     uint16 logits[T*V] (bf16 bits), int32 target[T], float old_logp[T], float adv[T],
 *     uint8 mask[T]
 * out: int32 status of the finish, float loss_tok[T], float logp_tok[T],
 *     uint16 dlogits[T*V], double loss, int64 n_valid, int64 n_clipped */
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

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: loss_step <in> <out>\n");
    return 1;
  }
  FILE* fi = fopen(argv[1], "rb");
  if (!fi) return 1;
  int64_t T = 0, V = 0;
  float eps = 0.f, scale = 0.f;
  if (!read_all(fi, &T, 8) || !read_all(fi, &V, 8) || !read_all(fi, &eps, 4) || !read_all(fi, &scale, 4)) return 1;
  const size_t nz = (size_t)T * (size_t)V;
  uint16_t* z = malloc(nz * 2);
  int32_t* tgt = malloc((size_t)T * 4);
  float* old = malloc((size_t)T * 4);
  float* adv = malloc((size_t)T * 4);
  uint8_t* mask = malloc((size_t)T);
  if (!z || !tgt || !old || !adv || !mask) return 1;
  if (!read_all(fi, z, nz * 2) || !read_all(fi, tgt, (size_t)T * 4) || !read_all(fi, old, (size_t)T * 4) ||
      !read_all(fi, adv, (size_t)T * 4) || !read_all(fi, mask, (size_t)T))
    return 1;
  fclose(fi);

  void *d_z, *d_dz, *d_tgt, *d_old, *d_adv, *d_mask, *d_loss, *d_logp, *d_acc;
  CK(cudaMalloc(&d_z, nz * 2));
  CK(cudaMalloc(&d_dz, nz * 2));
  CK(cudaMalloc(&d_tgt, (size_t)T * 4));
  CK(cudaMalloc(&d_old, (size_t)T * 4));
  CK(cudaMalloc(&d_adv, (size_t)T * 4));
  CK(cudaMalloc(&d_mask, (size_t)T));
  CK(cudaMalloc(&d_loss, (size_t)T * 4));
  CK(cudaMalloc(&d_logp, (size_t)T * 4));
  CK(cudaMalloc(&d_acc, sizeof(grpo_step_acc)));
  CK(cudaMemset(d_acc, 0, sizeof(grpo_step_acc)));
  CK(cudaMemcpy(d_z, z, nz * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_tgt, tgt, (size_t)T * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_old, old, (size_t)T * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_adv, adv, (size_t)T * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_mask, mask, (size_t)T, cudaMemcpyHostToDevice));

  int rc = grpo_logprob_loss_fwd_bwd(d_z, GRPO_DTYPE_BF16, T, V, V, NULL, d_tgt, d_old, d_adv, d_mask, eps, scale,
                                     d_dz, V, d_loss, d_logp, d_acc, NULL);
  if (rc != GRPO_OK) {
    fprintf(stderr, "grpo_logprob_loss_fwd_bwd: %s\n", grpo_status_string(rc));
    return 3;
  }
  grpo_step_result res;
  const int st = grpo_finish_step(d_acc, d_loss, T, -1, 0, NULL, NULL, NULL, 0, &res, NULL);
  if (st < 0 && st != GRPO_ERR_N_MISMATCH) {
    fprintf(stderr, "grpo_finish_step: %s\n", grpo_status_string(st));
    return 3;
  }
  float* loss = malloc((size_t)T * 4);
  float* logp = malloc((size_t)T * 4);
  if (!loss || !logp) return 1;
  CK(cudaMemcpy(loss, d_loss, (size_t)T * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(logp, d_logp, (size_t)T * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(z, d_dz, nz * 2, cudaMemcpyDeviceToHost));

  FILE* fo = fopen(argv[2], "wb");
  if (!fo) return 1;
  const int32_t status = st;
  if (!write_all(fo, &status, 4) || !write_all(fo, loss, (size_t)T * 4) || !write_all(fo, logp, (size_t)T * 4) ||
      !write_all(fo, z, nz * 2) || !write_all(fo, &res.loss, 8) || !write_all(fo, &res.n_valid, 8) ||
      !write_all(fo, &res.n_clipped, 8))
    return 1;
  fclose(fo);
  printf("loss %.9g n_valid %lld status %d\n", res.loss, (long long)res.n_valid, status);
  return 0;
}
