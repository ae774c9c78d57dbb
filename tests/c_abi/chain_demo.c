/*
 * chain_demo.c -- the C ABI from plain C, without Python or PyTorch:
 * y = relu(a + b) * 0.5 on 2^20 + 7 floats (vectors, remainder and tail),
 * device memory from the CUDA runtime, the fused launch on the legacy
 * default stream, and a bit-exact check against the same expression in C
 * (one fp32 addition, then relu and a halving, which are exact).
 *
 * Exit status: 0 ok (or no device: compiled and handled cleanly), 1 wrong
 * result, 2 an ABI call failed.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fuse.h"

static float next_value(uint32_t* s) {
  *s = *s * 1664525u + 1013904223u;          /* LCG */
  return ((float)(*s >> 8) / 16777216.0f) * 2.0f - 1.0f; /* [-1, 1) */
}

int main(void) {
  const int64_t n = (1 << 20) + 7;
  fuse_handle h;
  int rc = fuse_compile("add;relu;scale:0.5", &n, 1, FUSE_F32, &h);
  if (rc != FUSE_OK) {
    fprintf(stderr, "fuse_compile: %d %s\n", rc, fuse_last_error());
    return 2;
  }
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
    printf("compiled; no CUDA device here\n");
    fuse_release(h);
    return 0;
  }
  size_t bytes = (size_t)n * sizeof(float);
  float *ha = malloc(bytes), *hb = malloc(bytes), *hy = malloc(bytes);
  uint32_t s = 12345u;
  for (int64_t i = 0; i < n; ++i) {
    ha[i] = next_value(&s);
    hb[i] = next_value(&s);
  }
  float *da, *db, *dy;
  if (cudaMalloc((void**)&da, bytes) || cudaMalloc((void**)&db, bytes) ||
      cudaMalloc((void**)&dy, bytes)) {
    fprintf(stderr, "cudaMalloc failed\n");
    return 2;
  }
  cudaMemcpy(da, ha, bytes, cudaMemcpyHostToDevice);
  cudaMemcpy(db, hb, bytes, cudaMemcpyHostToDevice);
  const void* ins[2] = {da, db};
  rc = fuse_launch(h, ins, 2, dy, NULL);
  if (rc != FUSE_OK) {
    fprintf(stderr, "fuse_launch: %d %s\n", rc, fuse_last_error());
    return 2;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return 2;
  cudaMemcpy(hy, dy, bytes, cudaMemcpyDeviceToHost);
  int64_t bad = 0;
  for (int64_t i = 0; i < n; ++i) {
    float t = ha[i] + hb[i];
    t = t > 0.0f ? t : 0.0f;
    t *= 0.5f;
    if (memcmp(&t, &hy[i], sizeof t) != 0) ++bad;
  }
  int64_t launches = 0;
  fuse_stats(NULL, NULL, &launches, NULL);
  printf("%s: %lld of %lld elements differ, %lld launch(es)\n", bad ? "WRONG" : "ok",
         (long long)bad, (long long)n, (long long)launches);
  fuse_release(h);
  cudaFree(da);
  cudaFree(db);
  cudaFree(dy);
  free(ha);
  free(hb);
  free(hy);
  return bad ? 1 : 0;
}
