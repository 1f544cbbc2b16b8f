/*
 * A plain C program that uses libmhr_gemm.so through its C ABI alone
 * (include/mhr_gemm.h): device buffers from the CUDA runtime, one call of each
 * entry point, gemm_check() after each.  Test infrastructure: the inputs come
 * from files the caller writes, the outputs go to files the caller compares
 * with its reference.
 *
 *   gemm_from_c DIR M N K
 *
 * reads DIR/A.f32 (M x K) and DIR/B.f32 (K x N), row-major fp32, and writes
 * DIR/C_f32.f32, DIR/C_3xtf32.f32 and DIR/C_bf16.f32 (M x N).  The bf16 call
 * takes the operands' top 16 bits (exact for values that bf16 represents).
 * Exit status 0 on success; a message on stderr otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "mhr_gemm.h"

static int fail(const char* what, int code) {
  fprintf(stderr, "gemm_from_c: %s failed (%d)\n", what, code);
  return 1;
}

static int read_file(const char* dir, const char* name, void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return 0;
  const size_t got = fread(buf, 1, bytes, f);
  fclose(f);
  return got == bytes;
}

static int write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 0;
  const size_t put = fwrite(buf, 1, bytes, f);
  return fclose(f) == 0 && put == bytes;
}

int main(int argc, char** argv) {
  if (argc != 5) {
    fprintf(stderr, "usage: gemm_from_c DIR M N K\n");
    return 2;
  }
  const char* dir = argv[1];
  const int64_t M = atoll(argv[2]), N = atoll(argv[3]), K = atoll(argv[4]);
  const size_t a_n = (size_t)(M * K), b_n = (size_t)(K * N), c_n = (size_t)(M * N);
  float* a = malloc(a_n * 4);
  float* b = malloc(b_n * 4);
  float* c = malloc(c_n * 4);
  uint16_t* a16 = malloc(a_n * 2);
  uint16_t* b16 = malloc(b_n * 2);
  if (!a || !b || !c || !a16 || !b16) return fail("malloc", 0);
  if (!read_file(dir, "A.f32", a, a_n * 4) || !read_file(dir, "B.f32", b, b_n * 4))
    return fail("reading the inputs", 0);
  for (size_t i = 0; i < a_n; ++i) {
    uint32_t u;
    memcpy(&u, &a[i], 4);
    a16[i] = (uint16_t)(u >> 16);
  }
  for (size_t i = 0; i < b_n; ++i) {
    uint32_t u;
    memcpy(&u, &b[i], 4);
    b16[i] = (uint16_t)(u >> 16);
  }

  void *da, *db, *da16, *db16, *dc;
  if (cudaMalloc(&da, a_n * 4) || cudaMalloc(&db, b_n * 4) || cudaMalloc(&da16, a_n * 2) ||
      cudaMalloc(&db16, b_n * 2) || cudaMalloc(&dc, c_n * 4))
    return fail("cudaMalloc", 0);
  if (cudaMemcpy(da, a, a_n * 4, cudaMemcpyHostToDevice) ||
      cudaMemcpy(db, b, b_n * 4, cudaMemcpyHostToDevice) ||
      cudaMemcpy(da16, a16, a_n * 2, cudaMemcpyHostToDevice) ||
      cudaMemcpy(db16, b16, b_n * 2, cudaMemcpyHostToDevice))
    return fail("cudaMemcpy to the device", 0);

  int rc;
  if ((rc = gemm_f32(da, db, dc, M, N, K, K, N, N, NULL)) != MHR_OK) return fail("gemm_f32", rc);
  if ((rc = gemm_check(NULL)) != MHR_OK) return fail("gemm_check after gemm_f32", rc);
  if (cudaMemcpy(c, dc, c_n * 4, cudaMemcpyDeviceToHost)) return fail("cudaMemcpy back", 0);
  if (!write_file(dir, "C_f32.f32", c, c_n * 4)) return fail("writing C_f32", 0);

  if ((rc = gemm_f32_3xtf32(da, db, dc, M, N, K, K, N, N, NULL)) != MHR_OK)
    return fail("gemm_f32_3xtf32", rc);
  if ((rc = gemm_check(NULL)) != MHR_OK) return fail("gemm_check after gemm_f32_3xtf32", rc);
  if (cudaMemcpy(c, dc, c_n * 4, cudaMemcpyDeviceToHost)) return fail("cudaMemcpy back", 0);
  if (!write_file(dir, "C_3xtf32.f32", c, c_n * 4)) return fail("writing C_3xtf32", 0);

  if ((rc = gemm_bf16_f32acc(da16, db16, dc, M, N, K, K, N, N, NULL)) != MHR_OK)
    return fail("gemm_bf16_f32acc", rc);
  if ((rc = gemm_check(NULL)) != MHR_OK) return fail("gemm_check after gemm_bf16_f32acc", rc);
  if (cudaMemcpy(c, dc, c_n * 4, cudaMemcpyDeviceToHost)) return fail("cudaMemcpy back", 0);
  if (!write_file(dir, "C_bf16.f32", c, c_n * 4)) return fail("writing C_bf16", 0);

  printf("%s version %d: three entry points OK\n", gemm_status_string(MHR_OK), gemm_version());
  gemm_release();
  cudaFree(da);
  cudaFree(db);
  cudaFree(da16);
  cudaFree(db16);
  cudaFree(dc);
  free(a);
  free(b);
  free(c);
  free(a16);
  free(b16);
  return 0;
}
