/*
 * Plain C client of libswiglu on a GPU: reads A, W1, W2 (bf16 bit patterns)
 * from binary files, allocates device memory with the CUDA runtime, packs,
 * runs swiglu_forward, checks the device status and writes Y (bf16 bits).
 * No PyTorch anywhere. Usage: forward_from_c M K N a.bin w1.bin w2.bin y.bin
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "swiglu.h"

static void* read_file(const char* path, size_t bytes) {
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* p = malloc(bytes);
  if (p && fread(p, 1, bytes, f) != bytes) {
    free(p);
    p = NULL;
  }
  fclose(f);
  return p;
}

int main(int argc, char** argv) {
  if (argc != 8) {
    fprintf(stderr, "usage: %s M K N a.bin w1.bin w2.bin y.bin\n", argv[0]);
    return 2;
  }
  const int64_t M = atoll(argv[1]), K = atoll(argv[2]), N = atoll(argv[3]);
  const size_t a_bytes = (size_t)M * K * 2, w_bytes = (size_t)K * N * 2, y_bytes = (size_t)M * N * 2;
  void* a = read_file(argv[4], a_bytes);
  void* w1 = read_file(argv[5], w_bytes);
  void* w2 = read_file(argv[6], w_bytes);
  if (!a || !w1 || !w2) {
    fprintf(stderr, "cannot read the inputs\n");
    return 2;
  }
  const size_t wp_bytes = swiglu_packed_weight_bytes(K, N);
  void *da, *dw1, *dw2, *dwp, *dy;
  if (cudaMalloc(&da, a_bytes) || cudaMalloc(&dw1, w_bytes) || cudaMalloc(&dw2, w_bytes) ||
      cudaMalloc(&dwp, wp_bytes) || cudaMalloc(&dy, y_bytes)) {
    fprintf(stderr, "cudaMalloc failed\n");
    return 3;
  }
  cudaMemcpy(da, a, a_bytes, cudaMemcpyHostToDevice);
  cudaMemcpy(dw1, w1, w_bytes, cudaMemcpyHostToDevice);
  cudaMemcpy(dw2, w2, w_bytes, cudaMemcpyHostToDevice);
  swiglu_status_t st = swiglu_pack_weights(dw1, dw2, dwp, K, N, NULL);
  if (st == SWIGLU_OK) st = swiglu_forward(da, dwp, dy, M, K, N, NULL);
  if (st == SWIGLU_OK) st = swiglu_check_device_status(NULL);
  if (st != SWIGLU_OK) {
    fprintf(stderr, "libswiglu: %s\n", swiglu_status_string(st));
    return 4;
  }
  void* y = malloc(y_bytes);
  cudaMemcpy(y, dy, y_bytes, cudaMemcpyDeviceToHost);
  FILE* f = fopen(argv[7], "wb");
  if (!f || fwrite(y, 1, y_bytes, f) != y_bytes) return 5;
  fclose(f);
  char plan[256];
  swiglu_plan_string(M, K, N, 0, plan, sizeof plan);
  printf("%s\n", plan);
  return 0;
}
