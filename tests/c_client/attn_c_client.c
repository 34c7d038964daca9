/*
 * A plain C11 client of the attention library's C ABI (include/attn.h):
 * no C++, no framework.  With K = 0 every score is 0, so under the causal
 * mask row i averages V over keys 0..i: O_i = mean_{j<=i} V_j, LSE_i =
 * ln(i + 1), dQ = 0 exactly, and dV_j = sum_{i>=j} dO_i / (i + 1).  The
 * program checks these closed forms and exits 0 on success, 1 on a
 * mismatch, 2 on a library or CUDA error (3 with no usable device).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "attn.h"

static uint16_t f2bf(float f) { /* round to nearest even */
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static float bf2f(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

#define CK(x)                                                        \
  do {                                                               \
    cudaError_t e_ = (x);                                            \
    if (e_ != cudaSuccess) {                                         \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));       \
      return 2;                                                      \
    }                                                                \
  } while (0)

int main(void) {
  const int B = 2, H = 3, N = 300, d = 64;
  const size_t n = (size_t)B * N * H * d;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    printf("no device\n");
    return 3;
  }
  uint16_t *hv = malloc(n * 2), *hdo = malloc(n * 2), *hz = calloc(n, 2), *ho = malloc(n * 2),
           *hdq = malloc(n * 2), *hdv = malloc(n * 2);
  float* hl = malloc((size_t)B * H * N * 4);
  for (size_t i = 0; i < n; ++i) {
    hv[i] = f2bf((float)((i * 7919u) % 17) / 8.0f - 1.0f);  /* exact in bf16 */
    hdo[i] = f2bf((float)((i * 104729u) % 13) / 4.0f - 1.5f);
  }
  void *q, *k, *v, *o, *dO, *dq, *dk, *dv, *ws;
  float* lse;
  const size_t wsb = attn_bwd_workspace_size(B, H, N, d);
  CK(cudaMalloc(&q, n * 2)); CK(cudaMalloc(&k, n * 2)); CK(cudaMalloc(&v, n * 2));
  CK(cudaMalloc(&o, n * 2)); CK(cudaMalloc(&dO, n * 2)); CK(cudaMalloc(&dq, n * 2));
  CK(cudaMalloc(&dk, n * 2)); CK(cudaMalloc(&dv, n * 2)); CK(cudaMalloc(&ws, wsb));
  CK(cudaMalloc((void**)&lse, (size_t)B * H * N * 4));
  CK(cudaMemcpy(q, hv, n * 2, cudaMemcpyHostToDevice));  /* any Q: the scores are 0 */
  CK(cudaMemcpy(k, hz, n * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(v, hv, n * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dO, hdo, n * 2, cudaMemcpyHostToDevice));
  int rc = attn_fwd(q, k, v, o, lse, B, H, N, d, 0.125f, 1, ATTN_BF16, NULL);
  if (rc == ATTN_OK)
    rc = attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, 0.125f, 1, ATTN_BF16, ws, wsb, NULL);
  if (rc == ATTN_OK) rc = attn_status(NULL);
  if (rc != ATTN_OK) {
    fprintf(stderr, "attn error %d: %s\n", rc, attn_last_error_string());
    return 2;
  }
  CK(cudaMemcpy(ho, o, n * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(hdq, dq, n * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(hdv, dv, n * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(hl, lse, (size_t)B * H * N * 4, cudaMemcpyDeviceToHost));
  double eo = 0, el = 0, ev = 0, vmax = 0;
  int dq_nonzero = 0;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h)
      for (int c = 0; c < d; ++c) {
        double sum = 0.0, suffix = 0.0;
        for (int i = 0; i < N; ++i) { /* O_i = prefix mean of V */
          const size_t at = (((size_t)b * N + i) * H + h) * d + c;
          sum += bf2f(hv[at]);
          const double ref = sum / (i + 1);
          eo = fmax(eo, fabs(bf2f(ho[at]) - ref) - fabs(ref) / 256.0);
          if (bf2f(hdq[at]) != 0.0f) dq_nonzero = 1;
          if (c == 0) el = fmax(el, fabs(hl[((size_t)b * H + h) * N + i] - log(i + 1.0)));
        }
        for (int j = N - 1; j >= 0; --j) { /* dV_j = sum_{i>=j} dO_i / (i + 1) */
          const size_t at = (((size_t)b * N + j) * H + h) * d + c;
          suffix += bf2f(hdo[at]) / (j + 1);
          ev = fmax(ev, fabs(bf2f(hdv[at]) - suffix) - fabs(suffix) / 128.0);
          vmax = fmax(vmax, fabs(suffix));
        }
      }
  printf("O err beyond rounding %.3e, LSE err %.3e, dV err beyond rounding %.3e (|dV| <= %.2f), "
         "dQ all zero %s\n", eo, el, ev, vmax, dq_nonzero ? "no" : "yes");
  return (eo <= 1e-2 && el <= 1e-3 && ev <= 1e-2 && !dq_nonzero) ? 0 : 1;
}
