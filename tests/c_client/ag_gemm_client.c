/*
 * A plain C user of the library: nothing but include/ag_gemm.h, the CUDA
 * runtime and libaggemm.so.  It reads a problem from a directory, runs it
 * through the C ABI and writes the result back:
 *
 *   ag_gemm_client DIR
 *
 * DIR/meta.txt   "S R K N dtype" (dtype: 0 fp16, 1 int8, 2 bf16)
 * DIR/shardI.bin shard I, R x K (2-byte elements, or int8), row-major
 * DIR/B.bin      K x N
 * DIR/bias.bin, DIR/scale.bin   int8 only: N int32 / N fp32
 * writes DIR/C.bin (M x N fp32), or DIR/Ci.bin (M x N int32) and
 * DIR/D.bin (M x N fp16 bits).  Exit status 0 on success; on any failure the
 * library's (or the runtime's) message goes to stderr and the status is 1.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ag_gemm.h"

#define MAX_SHARDS 64

static int read_file(const char* dir, const char* name, void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) {
    fprintf(stderr, "cannot open %s\n", path);
    return 1;
  }
  const size_t got = fread(buf, 1, bytes, f);
  fclose(f);
  if (got != bytes) {
    fprintf(stderr, "%s: expected %zu bytes, read %zu\n", path, bytes, got);
    return 1;
  }
  return 0;
}

static int write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof(path), "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) {
    fprintf(stderr, "cannot create %s\n", path);
    return 1;
  }
  const size_t put = fwrite(buf, 1, bytes, f);
  fclose(f);
  return put == bytes ? 0 : 1;
}

#define CUDA_OK(call)                                                   \
  do {                                                                  \
    cudaError_t e_ = (call);                                            \
    if (e_ != cudaSuccess) {                                            \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));       \
      return 1;                                                         \
    }                                                                   \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s DIR\n", argv[0]);
    return 2;
  }
  const char* dir = argv[1];
  char meta_path[4096];
  snprintf(meta_path, sizeof(meta_path), "%s/meta.txt", dir);
  FILE* mf = fopen(meta_path, "r");
  if (!mf) {
    fprintf(stderr, "cannot open %s\n", meta_path);
    return 1;
  }
  int S = 0, dtype = 0;
  long long R = 0, K = 0, N = 0;
  const int n_read = fscanf(mf, "%d %lld %lld %lld %d", &S, &R, &K, &N, &dtype);
  fclose(mf);
  if (n_read != 5 || S < 1 || S > MAX_SHARDS || R < 1 || K < 1 || N < 1) {
    fprintf(stderr, "bad meta.txt\n");
    return 1;
  }
  const int64_t M = (int64_t)S * R;
  const size_t esz = dtype == AG_GEMM_I8 ? 1 : 2;

  /* host inputs */
  void* h_shard[MAX_SHARDS];
  void* d_shard[MAX_SHARDS];
  const void* shard_ptrs[MAX_SHARDS];
  for (int s = 0; s < S; ++s) {
    char name[64];
    snprintf(name, sizeof(name), "shard%d.bin", s);
    h_shard[s] = malloc((size_t)R * K * esz);
    if (!h_shard[s] || read_file(dir, name, h_shard[s], (size_t)R * K * esz)) return 1;
    CUDA_OK(cudaMalloc(&d_shard[s], (size_t)R * K * esz));
    CUDA_OK(cudaMemcpy(d_shard[s], h_shard[s], (size_t)R * K * esz, cudaMemcpyHostToDevice));
    shard_ptrs[s] = d_shard[s];
  }
  void* h_B = malloc((size_t)K * N * esz);
  void* d_B = NULL;
  if (!h_B || read_file(dir, "B.bin", h_B, (size_t)K * N * esz)) return 1;
  CUDA_OK(cudaMalloc(&d_B, (size_t)K * N * esz));
  CUDA_OK(cudaMemcpy(d_B, h_B, (size_t)K * N * esz, cudaMemcpyHostToDevice));

  cudaStream_t stream;
  CUDA_OK(cudaStreamCreate(&stream));
  ag_gemm_plan* plan = ag_gemm_plan_create(S, M, K, N, dtype, 0);
  if (!plan) {
    fprintf(stderr, "ag_gemm_plan_create: %s\n", ag_gemm_last_error_message());
    return 1;
  }

  int rc;
  if (dtype == AG_GEMM_I8) {
    int32_t* h_bias = (int32_t*)malloc((size_t)N * 4);
    float* h_scale = (float*)malloc((size_t)N * 4);
    if (!h_bias || !h_scale || read_file(dir, "bias.bin", h_bias, (size_t)N * 4) ||
        read_file(dir, "scale.bin", h_scale, (size_t)N * 4))
      return 1;
    int32_t *d_bias, *d_Ci;
    float* d_scale;
    void* d_D;
    CUDA_OK(cudaMalloc((void**)&d_bias, (size_t)N * 4));
    CUDA_OK(cudaMalloc((void**)&d_scale, (size_t)N * 4));
    CUDA_OK(cudaMalloc((void**)&d_Ci, (size_t)M * N * 4));
    CUDA_OK(cudaMalloc(&d_D, (size_t)M * N * 2));
    CUDA_OK(cudaMemcpy(d_bias, h_bias, (size_t)N * 4, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(d_scale, h_scale, (size_t)N * 4, cudaMemcpyHostToDevice));
    rc = ag_gemm_dequant_run(plan, shard_ptrs, d_B, d_bias, d_scale, d_Ci, d_D, stream);
    if (rc == AG_GEMM_OK) rc = ag_gemm_plan_status(plan);
    if (rc != AG_GEMM_OK) {
      fprintf(stderr, "int8 run: %d %s\n", rc, ag_gemm_last_error_message());
      return 1;
    }
    int32_t* h_Ci = (int32_t*)malloc((size_t)M * N * 4);
    uint16_t* h_D = (uint16_t*)malloc((size_t)M * N * 2);
    if (!h_Ci || !h_D) return 1;
    CUDA_OK(cudaMemcpy(h_Ci, d_Ci, (size_t)M * N * 4, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(h_D, d_D, (size_t)M * N * 2, cudaMemcpyDeviceToHost));
    if (write_file(dir, "Ci.bin", h_Ci, (size_t)M * N * 4) ||
        write_file(dir, "D.bin", h_D, (size_t)M * N * 2))
      return 1;
  } else {
    float* d_C;
    CUDA_OK(cudaMalloc((void**)&d_C, (size_t)M * N * 4));
    rc = ag_gemm_run(plan, shard_ptrs, d_B, d_C, stream);
    if (rc == AG_GEMM_OK) rc = ag_gemm_plan_status(plan);
    if (rc != AG_GEMM_OK) {
      fprintf(stderr, "run: %d %s\n", rc, ag_gemm_last_error_message());
      return 1;
    }
    float* h_C = (float*)malloc((size_t)M * N * 4);
    if (!h_C) return 1;
    CUDA_OK(cudaMemcpy(h_C, d_C, (size_t)M * N * 4, cudaMemcpyDeviceToHost));
    if (write_file(dir, "C.bin", h_C, (size_t)M * N * 4)) return 1;
  }
  ag_gemm_plan_destroy(plan);
  CUDA_OK(cudaStreamDestroy(stream));
  printf("ok: S=%d M=%lld K=%lld N=%lld dtype=%d\n", S, (long long)M, K, N, dtype);
  return 0;
}
