/*
 * The library used from plain C, with nothing but rrs.h and the CUDA runtime:
 * device buffers from cudaMalloc, a softmax and a row sum on a stream, the
 * results copied back and written to a file for the test to compare with the
 * float64 oracle, and the argument errors the header promises.
 *
 *   abi_example <out-file> <M> <N>
 *
 * x[i, j] is drawn from a 64-bit linear congruential generator (the same
 * recipe the test reproduces) as a uniform value in [-8, 8).  The output file
 * holds x (M*N floats), then softmax(x) (M*N floats), then the row sums (M).
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "rrs.h"

static float next_uniform(uint64_t* state) {
  *state = *state * 6364136223846793005ULL + 1442695040888963407ULL;
  return (float)((double)(*state >> 40) / (double)(1ULL << 24) * 16.0 - 8.0);
}

static int fail(const char* what, int code) {
  fprintf(stderr, "%s: %d (%s) %s\n", what, code, rrs_status_string(code), rrs_last_error());
  return 1;
}

int main(int argc, char** argv) {
  if (argc != 4) {
    fprintf(stderr, "usage: %s <out-file> <M> <N>\n", argv[0]);
    return 2;
  }
  const int64_t M = atoll(argv[2]), N = atoll(argv[3]);
  const size_t n = (size_t)(M * N);
  float* hx = (float*)malloc(n * sizeof(float));
  float* hy = (float*)malloc(n * sizeof(float));
  float* hs = (float*)malloc((size_t)M * sizeof(float));
  if (!hx || !hy || !hs) return 2;
  uint64_t state = 12345;
  for (size_t i = 0; i < n; ++i) hx[i] = next_uniform(&state);

  float *dx = NULL, *dy = NULL, *ds = NULL;
  cudaStream_t stream;
  if (cudaMalloc((void**)&dx, n * sizeof(float)) != cudaSuccess ||
      cudaMalloc((void**)&dy, n * sizeof(float)) != cudaSuccess ||
      cudaMalloc((void**)&ds, (size_t)M * sizeof(float)) != cudaSuccess ||
      cudaStreamCreate(&stream) != cudaSuccess)
    return 3;
  cudaMemcpy(dx, hx, n * sizeof(float), cudaMemcpyHostToDevice);

  int st = softmax_rows(dx, dy, M, N, N, stream);
  if (st != RRS_OK) return fail("softmax_rows", st);
  st = row_sum(dx, ds, M, N, N, stream);
  if (st != RRS_OK) return fail("row_sum", st);
  st = rrs_device_error(stream);          /* synchronises the stream */
  if (st != RRS_OK) return fail("rrs_device_error", st);

  /* the errors the header promises, refused before anything is enqueued */
  if (softmax_rows(dx, dy, M, N, N - 1, stream) != RRS_ERR_INVALID_ARG) return fail("ld < N accepted", -1);
  if (softmax_rows(dx, dx + 1, M, N, N, stream) != RRS_ERR_ALIAS) return fail("overlap accepted", -1);
  if (softmax_rows(hx, dy, M, N, N, stream) != RRS_ERR_INVALID_ARG) return fail("host pointer accepted", -1);
  if (softmax_rows(dx, dy, 0, N, N, stream) != RRS_OK) return fail("empty call refused", -1);

  cudaMemcpy(hy, dy, n * sizeof(float), cudaMemcpyDeviceToHost);
  cudaMemcpy(hs, ds, (size_t)M * sizeof(float), cudaMemcpyDeviceToHost);
  FILE* f = fopen(argv[1], "wb");
  if (!f) return 4;
  fwrite(hx, sizeof(float), n, f);
  fwrite(hy, sizeof(float), n, f);
  fwrite(hs, sizeof(float), (size_t)M, f);
  fclose(f);
  cudaFree(dx);
  cudaFree(dy);
  cudaFree(ds);
  cudaStreamDestroy(stream);
  free(hx);
  free(hy);
  free(hs);
  printf("ok: version %d\n", rrs_version());
  return 0;
}
