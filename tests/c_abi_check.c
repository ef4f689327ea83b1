/* The C ABI used from plain C, without Python or torch: a small causal GQA
 * prefill and a split-KV decode through attn_fwd / attn_decode_splitkv on
 * device buffers from the CUDA runtime, checked against the fp64 oracle
 * (oracle_attn_rows from the test oracle's library) with the tolerance of
 * the parity tests.  Exit status 0 when every check passes. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "attn.h"

int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                     int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D, int causal,
                     double scale, const int64_t *rows, int64_t nrows, double *out_o,
                     double *out_lse, int nthreads);

static uint32_t g_state = 12345u;
/* bf16 bits of a pseudo-normal value (sum of four uniforms), round to nearest even */
static uint16_t rand_bf16(void) {
  float f = 0.f;
  for (int i = 0; i < 4; ++i) {
    g_state = g_state * 1664525u + 1013904223u;
    f += (float)(g_state >> 8) / 16777216.0f - 0.5f;
  }
  f *= 1.7320508f;
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

#define CHECK_CUDA(x)                                                   \
  do {                                                                  \
    cudaError_t e_ = (x);                                               \
    if (e_ != cudaSuccess) {                                            \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));          \
      return 2;                                                         \
    }                                                                   \
  } while (0)

/* |dO| <= 2e-2 absolute or relative per element, mean |dO| <= 2e-3, |dLSE| <= 1e-3 */
static int compare(const char *label, const uint16_t *o, const float *lse, const double *o_ref,
                   const double *lse_ref, int64_t rows, int64_t D) {
  double sum = 0.0, worst = 0.0, worst_lse = 0.0;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t d = 0; d < D; ++d) {
      const double ref = o_ref[r * D + d], err = fabs(bf16_value(o[r * D + d]) - ref);
      if (err > 2e-2 && err > 2e-2 * fabs(ref)) {
        fprintf(stderr, "%s: row %lld col %lld: %g vs %g\n", label, (long long)r, (long long)d,
                bf16_value(o[r * D + d]), ref);
        return 1;
      }
      sum += err;
      if (err > worst) worst = err;
    }
    const double el = fabs(lse[r] - lse_ref[r]);
    if (el > worst_lse) worst_lse = el;
  }
  const double mean = sum / (double)(rows * D);
  printf("%s: max |dO| %.3e, mean |dO| %.3e, max |dLSE| %.3e\n", label, worst, mean, worst_lse);
  return (mean <= 2e-3 && worst_lse <= 1e-3) ? 0 : 1;
}

int main(void) {
  /* prefill: causal, 4 query heads sharing 2 KV heads, ragged tails */
  const int B = 2, Hq = 4, Hkv = 2, Nq = 300, Nk = 300, D = 128;
  const float scale = 0.08838834764831845f;
  const size_t nq = (size_t)B * Hq * Nq * D, nkv = (size_t)B * Hkv * Nk * D;
  uint16_t *hq = malloc(nq * 2), *hk = malloc(nkv * 2), *hv = malloc(nkv * 2), *ho = malloc(nq * 2);
  float *hl = malloc((size_t)B * Hq * Nq * 4);
  double *o_ref = malloc(nq * 8), *l_ref = malloc((size_t)B * Hq * Nq * 8);
  if (!hq || !hk || !hv || !ho || !hl || !o_ref || !l_ref) return 2;
  for (size_t i = 0; i < nq; ++i) hq[i] = rand_bf16();
  for (size_t i = 0; i < nkv; ++i) hk[i] = rand_bf16();
  for (size_t i = 0; i < nkv; ++i) hv[i] = rand_bf16();

  void *dq, *dk, *dv, *dout;
  float *dl;
  CHECK_CUDA(cudaMalloc(&dq, nq * 2));
  CHECK_CUDA(cudaMalloc(&dk, nkv * 2));
  CHECK_CUDA(cudaMalloc(&dv, nkv * 2));
  CHECK_CUDA(cudaMalloc(&dout, nq * 2));
  CHECK_CUDA(cudaMalloc((void **)&dl, (size_t)B * Hq * Nq * 4));
  CHECK_CUDA(cudaMemcpy(dq, hq, nq * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dk, hk, nkv * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dv, hv, nkv * 2, cudaMemcpyHostToDevice));

  int rc = attn_fwd(dq, dk, dv, dout, dl, B, Hq, Hkv, Nq, Nk, D, 1, scale, 0);
  if (rc != ATTN_OK) {
    fprintf(stderr, "attn_fwd: %s\n", attn_status_string(rc));
    return 1;
  }
  /* invalid arguments come back as status codes, nothing launched */
  if (attn_fwd(dq, dk, dv, dout, dl, B, Hq, 3, Nq, Nk, D, 1, scale, 0) != ATTN_ERR_SHAPE) return 1;
  CHECK_CUDA(cudaDeviceSynchronize());
  CHECK_CUDA(cudaMemcpy(ho, dout, nq * 2, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(hl, dl, (size_t)B * Hq * Nq * 4, cudaMemcpyDeviceToHost));
  int64_t *rows = malloc((size_t)B * Hq * Nq * 8);
  if (!rows) return 2;
  for (int64_t r = 0; r < (int64_t)B * Hq * Nq; ++r) rows[r] = r;
  if (oracle_attn_rows(hq, hk, hv, B, Hq, Hkv, Nq, Nk, D, 1, (double)scale, rows,
                       (int64_t)B * Hq * Nq, o_ref, l_ref, 4) != 0)
    return 2;
  if (compare("prefill causal GQA", ho, hl, o_ref, l_ref, (int64_t)B * Hq * Nq, D)) return 1;

  /* decode: the first query row of each head against all Nk keys, 5 splits */
  uint16_t *hqd = malloc((size_t)B * Hq * D * 2);
  if (!hqd) return 2;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hq; ++h)
      memcpy(hqd + ((size_t)b * Hq + h) * D, hq + (((size_t)b * Hq + h) * Nq) * D, (size_t)D * 2);
  CHECK_CUDA(cudaMemcpy(dq, hqd, (size_t)B * Hq * D * 2, cudaMemcpyHostToDevice));
  rc = attn_decode_splitkv(dq, dk, dv, dout, dl, B, Hq, Hkv, Nk, D, 5, 0);
  if (rc != ATTN_OK) {
    fprintf(stderr, "attn_decode_splitkv: %s\n", attn_status_string(rc));
    return 1;
  }
  CHECK_CUDA(cudaDeviceSynchronize());
  CHECK_CUDA(cudaMemcpy(ho, dout, (size_t)B * Hq * D * 2, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(hl, dl, (size_t)B * Hq * 4, cudaMemcpyDeviceToHost));
  for (int64_t r = 0; r < (int64_t)B * Hq; ++r) rows[r] = r;
  if (oracle_attn_rows(hqd, hk, hv, B, Hq, Hkv, 1, Nk, D, 0, 1.0 / sqrt((double)D), rows,
                       (int64_t)B * Hq, o_ref, l_ref, 4) != 0)
    return 2;
  if (compare("decode split 5", ho, hl, o_ref, l_ref, (int64_t)B * Hq, D)) return 1;
  if (attn_get_device_error(0) != 0) return 1;
  printf("C ABI check passed\n");
  return 0;
}
