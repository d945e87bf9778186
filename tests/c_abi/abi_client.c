/*
 * A plain C client of libattnres (include/attnres.h): no Python, no torch.
 * Builds seeded bf16 inputs, runs one layer through attnres_aggregate on
 * device buffers and through attnres_aggregate_host on host buffers,
 * checks that the two agree bit for bit and that a bad argument is refused,
 * and writes inputs and outputs to a file for the oracle comparison done by
 * tests/test_gpu_c_abi.py.
 *
 *   abi_client OUT.bin        exit status 0 = every check passed
 *
 * File layout (little endian): int32 S, T, d; uint16 sources [S][T][d]
 * (bf16 bit patterns); float32 w [d]; uint16 r [T][d] (bf16); float32
 * weights [T][S].
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "attnres.h"

#define S_SRC 5
#define T_TOK 100
#define D_CH 7168

/* splitmix64: a counter-based stream for the inputs */
static uint64_t next_u64(uint64_t* x) {
  uint64_t z = (*x += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* a bf16 bit pattern with a random sign, exponent in [118, 129] (|x| in
 * [2^-9, 8)) and mantissa: always a finite normal number */
static uint16_t random_bf16(uint64_t* x) {
  const uint64_t r = next_u64(x);
  const uint16_t sign = (uint16_t)((r & 1u) << 15);
  const uint16_t expo = (uint16_t)(118u + (uint16_t)((r >> 1) % 12u));
  const uint16_t mant = (uint16_t)((r >> 8) & 0x7Fu);
  return (uint16_t)(sign | (uint16_t)(expo << 7) | mant);
}

#define CK(call)                                                            \
  do {                                                                      \
    cudaError_t e_ = (call);                                                \
    if (e_ != cudaSuccess) {                                                \
      fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));    \
      return 2;                                                             \
    }                                                                       \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s OUT.bin\n", argv[0]);
    return 2;
  }
  const size_t n_src = (size_t)S_SRC * T_TOK * D_CH, n_r = (size_t)T_TOK * D_CH, n_a = (size_t)T_TOK * S_SRC;
  uint16_t* h_src = (uint16_t*)malloc(n_src * 2);
  float* h_w = (float*)malloc(D_CH * 4);
  uint16_t* h_r = (uint16_t*)malloc(n_r * 2);
  uint16_t* h_r2 = (uint16_t*)malloc(n_r * 2);
  float* h_a = (float*)malloc(n_a * 4);
  float* h_a2 = (float*)malloc(n_a * 4);
  if (!h_src || !h_w || !h_r || !h_r2 || !h_a || !h_a2) return 2;
  uint64_t seed = 20261202u;
  for (size_t i = 0; i < n_src; ++i) h_src[i] = random_bf16(&seed);
  for (int c = 0; c < D_CH; ++c) h_w[c] = (float)((int64_t)(next_u64(&seed) >> 40) - (1 << 23)) / (float)(1 << 23) / 42.0f;

  /* device path */
  void *d_src, *d_r;
  float *d_w, *d_a;
  int* d_err;
  CK(cudaMalloc(&d_src, n_src * 2));
  CK(cudaMalloc((void**)&d_w, D_CH * 4));
  CK(cudaMalloc(&d_r, n_r * 2));
  CK(cudaMalloc((void**)&d_a, n_a * 4));
  CK(cudaMalloc((void**)&d_err, 4));
  CK(cudaMemcpy(d_src, h_src, n_src * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_w, h_w, D_CH * 4, cudaMemcpyHostToDevice));
  CK(cudaMemset(d_err, 0, 4));
  const void* srcs[S_SRC];
  for (int s = 0; s < S_SRC; ++s) srcs[s] = (const char*)d_src + (size_t)s * T_TOK * D_CH * 2;
  int rc = attnres_aggregate(srcs, S_SRC, T_TOK, D_CH, ATTNRES_BF16, d_w, ATTNRES_DEFAULT_EPS, d_r, ATTNRES_BF16,
                             d_a, d_err, NULL);
  if (rc != ATTNRES_OK) {
    fprintf(stderr, "attnres_aggregate: %s (%s)\n", attnres_status_string(rc), attnres_last_error());
    return 1;
  }
  CK(cudaDeviceSynchronize());
  int h_err = -1;
  CK(cudaMemcpy(&h_err, d_err, 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(h_r, d_r, n_r * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(h_a, d_a, n_a * 4, cudaMemcpyDeviceToHost));
  if (h_err != 0) {
    fprintf(stderr, "device error flags %d\n", h_err);
    return 1;
  }

  /* host-buffer path: 32-token chunks through 2 staging slots */
  const int64_t ws_bytes = attnres_aggregate_host_workspace_size(S_SRC, 32, D_CH, ATTNRES_BF16, ATTNRES_BF16, 1, 2);
  if (ws_bytes <= 0) return 1;
  void* d_ws;
  CK(cudaMalloc(&d_ws, (size_t)ws_bytes));
  const void* hsrcs[S_SRC];
  for (int s = 0; s < S_SRC; ++s) hsrcs[s] = h_src + (size_t)s * T_TOK * D_CH;
  memset(h_r2, 0xFF, n_r * 2);
  rc = attnres_aggregate_host(hsrcs, S_SRC, T_TOK, D_CH, ATTNRES_BF16, h_w, ATTNRES_DEFAULT_EPS, h_r2,
                              ATTNRES_BF16, h_a2, 32, d_ws, ws_bytes, NULL, NULL);
  if (rc != ATTNRES_OK) {
    fprintf(stderr, "attnres_aggregate_host: %s (%s)\n", attnres_status_string(rc), attnres_last_error());
    return 1;
  }
  CK(cudaDeviceSynchronize());
  if (memcmp(h_r, h_r2, n_r * 2) != 0 || memcmp(h_a, h_a2, n_a * 4) != 0) {
    fprintf(stderr, "host-buffer results differ from the device-buffer ones\n");
    return 1;
  }

  /* a rejected argument: nothing launched, a message left */
  rc = attnres_aggregate(srcs, 0, T_TOK, D_CH, ATTNRES_BF16, d_w, ATTNRES_DEFAULT_EPS, d_r, ATTNRES_BF16, d_a,
                         NULL, NULL);
  if (rc != ATTNRES_EINVAL || attnres_last_error()[0] == '\0') {
    fprintf(stderr, "S = 0 not refused (%d)\n", rc);
    return 1;
  }

  FILE* f = fopen(argv[1], "wb");
  if (!f) return 2;
  const int32_t dims[3] = {S_SRC, T_TOK, D_CH};
  int ok = fwrite(dims, 4, 3, f) == 3 && fwrite(h_src, 2, n_src, f) == n_src && fwrite(h_w, 4, D_CH, f) == D_CH &&
           fwrite(h_r, 2, n_r, f) == n_r && fwrite(h_a, 4, n_a, f) == n_a;
  fclose(f);
  cudaFree(d_src);
  cudaFree(d_w);
  cudaFree(d_r);
  cudaFree(d_a);
  cudaFree(d_err);
  cudaFree(d_ws);
  free(h_src);
  free(h_w);
  free(h_r);
  free(h_r2);
  free(h_a);
  free(h_a2);
  if (!ok) return 2;
  printf("c abi client ok: S=%d T=%d d=%d\n", S_SRC, T_TOK, D_CH);
  return 0;
}
