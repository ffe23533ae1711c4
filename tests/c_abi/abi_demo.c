/*
 * abi_demo.c - the MoE layer driven from plain C through include/moe.h and the CUDA runtime only (no Python, no
 * torch): the calling sequence a C or C++ host program uses.
 *
 *   abi_demo host   queries and host-side validation only (no device work; runs without a GPU)
 *   abi_demo run    routing, forward and backward of a small layer on device buffers from cudaMalloc; checks
 *                   the status codes, P = T*K under token choice, the device status word, and that O and dX are
 *                   finite and not all zero
 * Exit code 0 on success; a message on stderr otherwise.
 */
#include <cuda_runtime_api.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "moe.h"

#define CHECK(call)                                                                         \
  do {                                                                                      \
    int rc_ = (call);                                                                       \
    if (rc_ != MOE_OK) {                                                                    \
      fprintf(stderr, "%s:%d: %s -> %d (%s)\n", __FILE__, __LINE__, #call, rc_, moe_strerror(rc_)); \
      return 1;                                                                             \
    }                                                                                       \
  } while (0)
#define CUDA(call)                                                                          \
  do {                                                                                      \
    cudaError_t e_ = (call);                                                                \
    if (e_ != cudaSuccess) {                                                                \
      fprintf(stderr, "%s:%d: %s -> %s\n", __FILE__, __LINE__, #call, cudaGetErrorString(e_)); \
      return 1;                                                                             \
    }                                                                                       \
  } while (0)

enum { T = 512, D = 256, N = 128, E = 8, K = 2 };

static uint16_t to_bf16(float f) { /* round to nearest even */
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* a small deterministic pseudo-random value in [-1, 1) (64-bit LCG) */
static float rnd(uint64_t *s) {
  *s = *s * 6364136223846793005ull + 1442695040888963407ull;
  return (float)((*s >> 40) & 0xffffffu) / 8388608.0f - 1.0f;
}

static int host_checks(void) {
  size_t cap = 0, ws = 0;
  CHECK(moe_route_capacity(T, E, K, MOE_ROUTE_TC, &cap));
  if (cap != (size_t)T * K) return fprintf(stderr, "capacity %zu\n", cap), 1;
  CHECK(moe_route_capacity(T, E, K, MOE_ROUTE_TR, &cap));
  if (cap != (size_t)T * K + (size_t)E * (MOE_M_TILE / 2)) return fprintf(stderr, "TR capacity %zu\n", cap), 1;
  CHECK(moe_route_workspace_size(T, E, K, MOE_ROUTE_EC, &ws));
  CHECK(moe_forward_workspace_size_ex(T, D, N, E, K, (size_t)T * K, MOE_FLAG_DETERMINISTIC, &ws));
  if (moe_route_capacity(T, E, E + 1, MOE_ROUTE_TC, &cap) != MOE_ERR_INVALID_ARG) return 1;
  if (moe_forward_workspace_size(T, 200, N, E, K, (size_t)T * K, &ws) != MOE_ERR_UNSUPPORTED_SHAPE) return 1;
  if (moe_forward_workspace_size_ex(T, D, N, E, K, (size_t)T * K, 4u, &ws) != MOE_ERR_INVALID_ARG) return 1;
  if (strcmp(moe_strerror(MOE_ERR_WORKSPACE), "workspace missing or too small") != 0) return 1;
  printf("host checks ok\n");
  return 0;
}

static int run(void) {
  size_t cap = 0, ws_r = 0, ws_f = 0, ws_b = 0;
  CHECK(moe_route_capacity(T, E, K, MOE_ROUTE_TC, &cap));
  CHECK(moe_route_workspace_size(T, E, K, MOE_ROUTE_TC, &ws_r));
  CHECK(moe_forward_workspace_size(T, D, N, E, K, cap, &ws_f));
  CHECK(moe_backward_workspace_size(T, D, N, E, K, cap, &ws_b));

  /* inputs on the host: logits ~ U(-1, 1), X, dO ~ U(-1, 1), W1 ~ U(-1, 1)/sqrt(d), W2 ~ U(-1, 1)/sqrt(n) */
  uint64_t seed = 12345u;
  float *z = malloc(sizeof(float) * T * E);
  uint16_t *x = malloc(2 * (size_t)T * D), *dout = malloc(2 * (size_t)T * D);
  uint16_t *w1 = malloc(2 * (size_t)E * D * 2 * N), *w2 = malloc(2 * (size_t)E * N * D);
  for (size_t i = 0; i < (size_t)T * E; ++i) z[i] = rnd(&seed);
  for (size_t i = 0; i < (size_t)T * D; ++i) x[i] = to_bf16(rnd(&seed));
  for (size_t i = 0; i < (size_t)E * D * 2 * N; ++i) w1[i] = to_bf16(rnd(&seed) / 16.0f);
  for (size_t i = 0; i < (size_t)E * N * D; ++i) w2[i] = to_bf16(rnd(&seed) / 11.3f);
  for (size_t i = 0; i < (size_t)T * D; ++i) dout[i] = to_bf16(rnd(&seed));

  /* device buffers, all owned here */
  float *d_z, *d_topk_score, *d_row_score, *d_ds;
  int32_t *d_topk_idx, *d_tc, *d_counts, *d_off, *d_toff, *d_row_token, *d_row_slot, *d_status;
  uint16_t *d_x, *d_w1, *d_w2, *d_do, *d_o, *d_h, *d_dx, *d_dw1, *d_dw2;
  void *d_ws_r, *d_ws_f, *d_ws_b;
  CUDA(cudaMalloc((void **)&d_z, sizeof(float) * T * E));
  CUDA(cudaMalloc((void **)&d_topk_idx, 4 * T * K));
  CUDA(cudaMalloc((void **)&d_topk_score, 4 * T * K));
  CUDA(cudaMalloc((void **)&d_tc, 4 * E));
  CUDA(cudaMalloc((void **)&d_counts, 4 * E));
  CUDA(cudaMalloc((void **)&d_off, 4 * (E + 1)));
  CUDA(cudaMalloc((void **)&d_toff, 4 * (E + 1)));
  CUDA(cudaMalloc((void **)&d_row_token, 4 * cap));
  CUDA(cudaMalloc((void **)&d_row_slot, 4 * cap));
  CUDA(cudaMalloc((void **)&d_row_score, 4 * cap));
  CUDA(cudaMalloc((void **)&d_status, 4 * MOE_STATUS_WORDS));
  CUDA(cudaMalloc((void **)&d_x, 2 * (size_t)T * D));
  CUDA(cudaMalloc((void **)&d_do, 2 * (size_t)T * D));
  CUDA(cudaMalloc((void **)&d_w1, 2 * (size_t)E * D * 2 * N));
  CUDA(cudaMalloc((void **)&d_w2, 2 * (size_t)E * N * D));
  CUDA(cudaMalloc((void **)&d_o, 2 * (size_t)T * D));
  CUDA(cudaMalloc((void **)&d_h, 2 * cap * 2 * N));
  CUDA(cudaMalloc((void **)&d_dx, 2 * (size_t)T * D));
  CUDA(cudaMalloc((void **)&d_dw1, 2 * (size_t)E * D * 2 * N));
  CUDA(cudaMalloc((void **)&d_dw2, 2 * (size_t)E * N * D));
  CUDA(cudaMalloc((void **)&d_ds, 4 * cap));
  CUDA(cudaMalloc(&d_ws_r, ws_r));
  CUDA(cudaMalloc(&d_ws_f, ws_f));
  CUDA(cudaMalloc(&d_ws_b, ws_b));
  CUDA(cudaMemcpy(d_z, z, sizeof(float) * T * E, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_x, x, 2 * (size_t)T * D, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_do, dout, 2 * (size_t)T * D, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_w1, w1, 2 * (size_t)E * D * 2 * N, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_w2, w2, 2 * (size_t)E * N * D, cudaMemcpyHostToDevice));

  cudaStream_t s;
  CUDA(cudaStreamCreate(&s));
  moe_routing r = {d_topk_idx, d_topk_score, d_tc, d_counts, d_off, d_toff, d_row_token, d_row_slot, d_row_score,
                   d_status};
  int32_t P = 0;
  CHECK(moe_route(d_z, T, E, K, MOE_ROUTE_TC, &r, d_ws_r, ws_r, &P, s));
  if (P != T * K) return fprintf(stderr, "P = %d, expected %d\n", P, T * K), 1;
  CHECK(moe_forward(d_x, d_w1, d_w2, &r, T, D, N, E, K, cap, d_o, d_h, d_ws_f, ws_f, s));
  CHECK(moe_backward(d_do, d_x, d_w1, d_w2, d_h, &r, T, D, N, E, K, cap, d_dx, d_dw1, d_dw2, d_ds, d_ws_b, ws_b, s));
  int32_t code = -1, P2 = 0;
  CHECK(moe_get_status(&r, &code, &P2, s));
  if (code != MOE_OK || P2 != P) return fprintf(stderr, "device status %d, P %d\n", code, P2), 1;

  uint16_t *o = malloc(2 * (size_t)T * D), *dx = malloc(2 * (size_t)T * D);
  CUDA(cudaMemcpy(o, d_o, 2 * (size_t)T * D, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(dx, d_dx, 2 * (size_t)T * D, cudaMemcpyDeviceToHost));
  double so = 0.0, sdx = 0.0;
  for (size_t i = 0; i < (size_t)T * D; ++i) {
    const float a = from_bf16(o[i]), b = from_bf16(dx[i]);
    if (!isfinite(a) || !isfinite(b)) return fprintf(stderr, "non-finite output at %zu\n", i), 1;
    so += fabs(a);
    sdx += fabs(b);
  }
  if (so == 0.0 || sdx == 0.0) return fprintf(stderr, "all-zero output\n"), 1;
  printf("run ok: P = %d, mean |O| = %.4g, mean |dX| = %.4g, kernels launched %llu\n", P, so / (T * D),
         sdx / (T * D), (unsigned long long)moe_kernel_launch_count());
  CUDA(cudaStreamDestroy(s));
  return 0;
}

int main(int argc, char **argv) {
  if (argc > 1 && strcmp(argv[1], "run") == 0) return run();
  return host_checks();
}
