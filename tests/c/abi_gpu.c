/* The C ABI used from plain C on a GPU: an int32 allreduce of 4 simulated
 * ranks (ragged length) and an all-gather through libhoc, checked element by
 * element against sums computed here.  Device buffers come from cudaMalloc;
 * no Python, no PyTorch.  Exits 0 and prints "ABI GPU OK" when every element
 * matches. */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "hoc.h"

#define K 4
#define N 1000003

static int value(int r, size_t i) { return (int)((i * 7u + (size_t)r * 131u) % 1000u) - 500; }

int main(void) {
  hocComm_t comm = NULL;
  hocResult_t rc = hoc_init(&comm, K, 0, NULL);
  if (rc != HOC_SUCCESS) {
    printf("hoc_init: %s (%s)\n", hoc_error_string(rc), hoc_last_error_detail());
    return 1;
  }
  int* host = (int*)malloc(sizeof(int) * N);
  void* send[K];
  void* recv[K];
  void* gath[K];
  for (int r = 0; r < K; ++r) {
    for (size_t i = 0; i < N; ++i) host[i] = value(r, i);
    if (cudaMalloc(&send[r], sizeof(int) * N) != cudaSuccess || cudaMalloc(&recv[r], sizeof(int) * N) != cudaSuccess ||
        cudaMalloc(&gath[r], sizeof(int) * N * K) != cudaSuccess) {
      printf("cudaMalloc failed\n");
      return 1;
    }
    cudaMemcpy(send[r], host, sizeof(int) * N, cudaMemcpyHostToDevice);
  }
  rc = hoc_allreduce(comm, (const void* const*)send, recv, N, HOC_INT32, HOC_SUM, NULL);
  if (rc == HOC_SUCCESS) rc = hoc_allgather(comm, (const void* const*)send, gath, N, HOC_INT32, NULL);
  if (rc == HOC_SUCCESS) rc = hoc_wait(comm, NULL, 30000);
  if (rc != HOC_SUCCESS) {
    printf("collective: %s (%s)\n", hoc_error_string(rc), hoc_last_error_detail());
    return 1;
  }
  int* out = (int*)malloc(sizeof(int) * N * K);
  for (int r = 0; r < K; ++r) {
    cudaMemcpy(host, recv[r], sizeof(int) * N, cudaMemcpyDeviceToHost);
    for (size_t i = 0; i < N; ++i) {
      int want = 0;
      for (int q = 0; q < K; ++q) want += value(q, i);
      if (host[i] != want) {
        printf("allreduce rank %d element %zu: %d, want %d\n", r, i, host[i], want);
        return 1;
      }
    }
    cudaMemcpy(out, gath[r], sizeof(int) * N * K, cudaMemcpyDeviceToHost);
    for (int q = 0; q < K; ++q)
      for (size_t i = 0; i < N; ++i)
        if (out[(size_t)q * N + i] != value(q, i)) {
          printf("allgather rank %d block %d element %zu: %d, want %d\n", r, q, i, out[(size_t)q * N + i], value(q, i));
          return 1;
        }
  }
  for (int r = 0; r < K; ++r) {
    cudaFree(send[r]);
    cudaFree(recv[r]);
    cudaFree(gath[r]);
  }
  free(host);
  free(out);
  if (hoc_destroy(comm) != HOC_SUCCESS) return 1;
  printf("ABI GPU OK\n");
  return 0;
}
