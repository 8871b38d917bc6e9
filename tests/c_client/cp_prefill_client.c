/*
 * A plain C client of libslope (no Python, no torch): device buffers from the CUDA runtime,
 * deterministic bf16 inputs, then the context-parallel prefill (zigzag ring of 4) and the
 * same attention as one launch over the whole sequence, which must agree within the bf16
 * output tolerance.  Also checks an argument error and the device status word.
 * Prints "ok <max abs difference>" and exits 0 on success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "slope.h"

#define S 2048
#define HQ 8
#define HKV 2
#define D 64

static uint16_t to_bf16(float x) { /* round to nearest even (finite inputs) */
  uint32_t u;
  memcpy(&u, &x, 4);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
static float from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float x;
  memcpy(&x, &u, 4);
  return x;
}
static slope_tensor desc(void* data, slope_dtype dt, int64_t a, int64_t b, int64_t c) {
  slope_tensor t;
  memset(&t, 0, sizeof(t));
  t.data = data;
  t.dtype = dt;
  t.ndim = 3;
  t.shape[0] = a;
  t.shape[1] = b;
  t.shape[2] = c;
  t.stride[0] = b * c;
  t.stride[1] = c;
  t.stride[2] = 1;
  return t;
}
#define CHECK(x)                                                    \
  do {                                                              \
    if (!(x)) {                                                     \
      fprintf(stderr, "check failed: %s (line %d)\n", #x, __LINE__); \
      return 1;                                                     \
    }                                                               \
  } while (0)

int main(void) {
  const size_t nq = (size_t)S * HQ * D, nkv = (size_t)S * HKV * D;
  uint16_t* hq = malloc(nq * 2);
  uint16_t* hk = malloc(nkv * 2);
  uint16_t* hv = malloc(nkv * 2);
  uint16_t* o1 = malloc(nq * 2);
  uint16_t* o2 = malloc(nq * 2);
  CHECK(hq && hk && hv && o1 && o2);
  uint32_t seed = 12345u;
  for (size_t i = 0; i < nq; ++i) {
    seed = seed * 1664525u + 1013904223u;
    hq[i] = to_bf16(((float)(seed >> 8) / 16777216.0f - 0.5f) * 2.0f);
  }
  for (size_t i = 0; i < nkv; ++i) {
    seed = seed * 1664525u + 1013904223u;
    hk[i] = to_bf16(((float)(seed >> 8) / 16777216.0f - 0.5f) * 2.0f);
    seed = seed * 1664525u + 1013904223u;
    hv[i] = to_bf16(((float)(seed >> 8) / 16777216.0f - 0.5f) * 2.0f);
  }
  void *dq, *dk, *dv, *do1, *do2, *dl1, *dl2, *ws;
  const size_t ws_bytes = slope_cp_prefill_workspace_size(S, HQ, D, 4, SLOPE_LAYOUT_ZIGZAG, NULL);
  CHECK(ws_bytes > 0);
  CHECK(cudaMalloc(&dq, nq * 2) == cudaSuccess && cudaMalloc(&dk, nkv * 2) == cudaSuccess &&
        cudaMalloc(&dv, nkv * 2) == cudaSuccess && cudaMalloc(&do1, nq * 2) == cudaSuccess &&
        cudaMalloc(&do2, nq * 2) == cudaSuccess && cudaMalloc(&dl1, (size_t)HQ * S * 4) == cudaSuccess &&
        cudaMalloc(&dl2, (size_t)HQ * S * 4) == cudaSuccess && cudaMalloc(&ws, ws_bytes) == cudaSuccess);
  CHECK(cudaMemcpy(dq, hq, nq * 2, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemcpy(dk, hk, nkv * 2, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemcpy(dv, hv, nkv * 2, cudaMemcpyHostToDevice) == cudaSuccess);

  slope_tensor q = desc(dq, SLOPE_BF16, S, HQ, D), k = desc(dk, SLOPE_BF16, S, HKV, D);
  slope_tensor v = desc(dv, SLOPE_BF16, S, HKV, D);
  slope_tensor out1 = desc(do1, SLOPE_BF16, S, HQ, D), out2 = desc(do2, SLOPE_BF16, S, HQ, D);
  slope_tensor lse1, lse2;
  memset(&lse1, 0, sizeof(lse1));
  lse1.data = dl1;
  lse1.dtype = SLOPE_F32;
  lse1.ndim = 2;
  lse1.shape[0] = HQ;
  lse1.shape[1] = S;
  lse1.stride[0] = S;
  lse1.stride[1] = 1;
  lse2 = lse1;
  lse2.data = dl2;

  /* an argument error is reported before any launch */
  CHECK(slope_cp_prefill(&q, &k, &v, 3, SLOPE_LAYOUT_ZIGZAG, NULL, 1, 0, 0.0f, &out1, &lse1, ws, ws_bytes, NULL) ==
        SLOPE_ERR_LAYOUT);
  CHECK(slope_cp_prefill(&q, &k, &v, 4, SLOPE_LAYOUT_ZIGZAG, NULL, 1, 0, 0.0f, &out1, &lse1, ws, ws_bytes, NULL) ==
        SLOPE_OK);
  CHECK(slope_attn_partial(&q, &k, &v, 0, 0, 1, 0, 0.0f, &out2, &lse2, NULL) == SLOPE_OK);
  int site = -1;
  CHECK(slope_device_status(NULL, &site) == SLOPE_OK && site == 0);
  CHECK(cudaMemcpy(o1, do1, nq * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(cudaMemcpy(o2, do2, nq * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
  double worst = 0.0;
  for (size_t i = 0; i < nq; ++i) {
    const double a = from_bf16(o1[i]), b = from_bf16(o2[i]);
    CHECK(isfinite(a) && isfinite(b));
    if (fabs(a - b) > worst) worst = fabs(a - b);
  }
  CHECK(worst <= 2e-2);
  /* the log-sum-exps of both calls: finite (every causal row sees itself) and within 1e-3 */
  float* l1 = malloc((size_t)HQ * S * 4);
  float* l2 = malloc((size_t)HQ * S * 4);
  CHECK(l1 && l2);
  CHECK(cudaMemcpy(l1, dl1, (size_t)HQ * S * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(cudaMemcpy(l2, dl2, (size_t)HQ * S * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  double worst_lse = 0.0;
  for (size_t i = 0; i < (size_t)HQ * S; ++i) {
    CHECK(isfinite(l1[i]) && isfinite(l2[i]));
    if (fabs((double)l1[i] - (double)l2[i]) > worst_lse) worst_lse = fabs((double)l1[i] - (double)l2[i]);
  }
  CHECK(worst_lse <= 1e-3);
  free(l1);
  free(l2);
  printf("ok %.3e %.3e %s\n", worst, worst_lse, slope_version());
  cudaFree(dq);
  cudaFree(dk);
  cudaFree(dv);
  cudaFree(do1);
  cudaFree(do2);
  cudaFree(dl1);
  cudaFree(dl2);
  cudaFree(ws);
  free(hq);
  free(hk);
  free(hv);
  free(o1);
  free(o2);
  return 0;
}
