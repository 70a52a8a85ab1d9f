/*
 * The C ABI of libmoe.so used from plain C (no Python, no torch): allocate device buffers with
 * the CUDA runtime, run one MoE layer forward and its backward on a small seeded problem, and
 * print a checksum line that the calling test compares with the same computation made through
 * the Python binding (the inputs are written as raw bf16 files to the directory given as the
 * first argument).  Exit status 0 on success.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "moe.h"

#define CHECK_CUDA(x)                                                            \
  do {                                                                           \
    cudaError_t e_ = (x);                                                        \
    if (e_ != cudaSuccess) {                                                     \
      fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));          \
      return 2;                                                                  \
    }                                                                            \
  } while (0)
#define CHECK_MOE(x)                                                             \
  do {                                                                           \
    moe_status s_ = (x);                                                         \
    if (s_ != MOE_OK) {                                                          \
      fprintf(stderr, "%s failed: %s\n", #x, moe_status_string(s_));           \
      return 3;                                                                  \
    }                                                                            \
  } while (0)

/* bf16 bit patterns of a few small deterministic values (exactly representable) */
static uint16_t bf16_of(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  return (uint16_t)(u >> 16);
}
static float f32_of(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float v;
  memcpy(&v, &u, 4);
  return v;
}

static void fill(uint16_t* a, size_t count, uint32_t seed, float scale) {
  uint32_t s = seed * 2654435761u + 12345u;
  for (size_t i = 0; i < count; ++i) {
    s = s * 1664525u + 1013904223u;
    const int v = (int)((s >> 9) & 0xFF) - 128; /* -128 .. 127 */
    a[i] = bf16_of(scale * (float)v / 128.0f);
  }
}

static int dump(const char* dir, const char* name, const void* p, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s.bin", dir, name);
  FILE* fh = fopen(path, "wb");
  if (!fh) return 1;
  const size_t w = fwrite(p, 1, bytes, fh);
  fclose(fh);
  return w == bytes ? 0 : 1;
}

int main(int argc, char** argv) {
  const int T = 200, d = 256, f = 384, n = 8, k = 2;
  const size_t nx = (size_t)T * d, nw1 = (size_t)n * f * d, nwg = (size_t)d * n;
  uint16_t *hx = malloc(nx * 2), *hdy = malloc(nx * 2), *hwg = malloc(nwg * 2);
  uint16_t *hw1 = malloc(nw1 * 2), *hw3 = malloc(nw1 * 2), *hw2 = malloc(nw1 * 2);
  fill(hx, nx, 1, 1.0f);
  fill(hdy, nx, 2, 1.0f);
  fill(hwg, nwg, 3, 0.05f);
  fill(hw1, nw1, 4, 0.0625f);
  fill(hw3, nw1, 5, 0.0625f);
  fill(hw2, nw1, 6, 0.05f);
  if (argc > 1) {
    /* the inputs, for the caller to run the same layer through the Python binding */
    if (dump(argv[1], "x", hx, nx * 2) || dump(argv[1], "dy", hdy, nx * 2) ||
        dump(argv[1], "wg", hwg, nwg * 2) || dump(argv[1], "w1", hw1, nw1 * 2) ||
        dump(argv[1], "w3", hw3, nw1 * 2) || dump(argv[1], "w2", hw2, nw1 * 2))
      return 5;
  }

  void *x, *dy, *wg, *w1, *w3, *w2, *y, *dx, *dw1, *dw3, *dw2, *ws, *bws;
  float* dwg;
  const size_t wsz = moe_workspace_size(T, d, f, n, k, MOE_BF16);
  const size_t bsz = moe_backward_workspace_size(T, d, f, n, k, MOE_BF16);
  if (wsz == 0 || bsz == 0) return 4;
  CHECK_CUDA(cudaMalloc(&x, nx * 2));
  CHECK_CUDA(cudaMalloc(&dy, nx * 2));
  CHECK_CUDA(cudaMalloc(&y, nx * 2));
  CHECK_CUDA(cudaMalloc(&dx, nx * 2));
  CHECK_CUDA(cudaMalloc(&wg, nwg * 2));
  CHECK_CUDA(cudaMalloc(&w1, nw1 * 2));
  CHECK_CUDA(cudaMalloc(&w3, nw1 * 2));
  CHECK_CUDA(cudaMalloc(&w2, nw1 * 2));
  CHECK_CUDA(cudaMalloc(&dw1, nw1 * 2));
  CHECK_CUDA(cudaMalloc(&dw3, nw1 * 2));
  CHECK_CUDA(cudaMalloc(&dw2, nw1 * 2));
  CHECK_CUDA(cudaMalloc((void**)&dwg, nwg * 4));
  CHECK_CUDA(cudaMalloc(&ws, wsz));
  CHECK_CUDA(cudaMalloc(&bws, bsz));
  CHECK_CUDA(cudaMemset(ws, 0, 256));
  CHECK_CUDA(cudaMemset(bws, 0, 256));
  CHECK_CUDA(cudaMemcpy(x, hx, nx * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(dy, hdy, nx * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(wg, hwg, nwg * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(w1, hw1, nw1 * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(w3, hw3, nw1 * 2, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(w2, hw2, nw1 * 2, cudaMemcpyHostToDevice));

  cudaStream_t s;
  CHECK_CUDA(cudaStreamCreate(&s));
  CHECK_MOE(moe_layer_forward(x, wg, NULL, w1, w3, w2, NULL, T, d, f, n, k, MOE_BF16, y, NULL,
                              NULL, ws, wsz, s));
  CHECK_MOE(moe_layer_backward(x, wg, NULL, w1, w3, w2, dy, T, d, f, n, k, MOE_BF16, dx, dwg, NULL,
                               dw1, dw3, dw2, bws, bsz, s));
  CHECK_MOE(moe_check_device_error(ws, wsz, s));
  CHECK_MOE(moe_check_device_error(bws, bsz, s));

  uint16_t* hy = malloc(nx * 2);
  uint16_t* hdw = malloc(nw1 * 2);
  float* hdwg = malloc(nwg * 4);
  CHECK_CUDA(cudaMemcpy(hy, y, nx * 2, cudaMemcpyDeviceToHost));
  double sy = 0, sdw = 0, sdwg = 0;
  for (size_t i = 0; i < nx; ++i) sy += fabs((double)f32_of(hy[i]));
  CHECK_CUDA(cudaMemcpy(hdw, dw2, nw1 * 2, cudaMemcpyDeviceToHost));
  for (size_t i = 0; i < nw1; ++i) sdw += fabs((double)f32_of(hdw[i]));
  CHECK_CUDA(cudaMemcpy(hdwg, dwg, nwg * 4, cudaMemcpyDeviceToHost));
  for (size_t i = 0; i < nwg; ++i) sdwg += fabs((double)hdwg[i]);
  /* checksums for the caller: sums of |y|, |dw2|, |dw_gate| */
  printf("version %d sum_abs_y %.9e sum_abs_dw2 %.9e sum_abs_dwg %.9e\n", moe_version(), sy, sdw,
         sdwg);
  CHECK_CUDA(cudaStreamDestroy(s));
  return 0;
}
