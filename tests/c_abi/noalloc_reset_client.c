/*
 * A plain C client of attnres_aggregate_backward_noalloc across a device
 * reset (no Python, no torch).  The entry point keeps its scratch in an
 * array built into the library and caches that array's device address; a
 * cudaDeviceReset tears the context down and the next context loads the
 * library's module again, possibly at another address, and without the
 * kernels' shared-memory opt-in.  The library keys both caches on the
 * context, so a call after the reset must give the very same gradients as
 * one before it.
 *
 *   noalloc_reset_client        exit status 0 = every check passed
 *
 * Checks: (1) before the reset, the no-alloc backward equals
 * attnres_aggregate_backward with a caller workspace bit for bit (same
 * kernels, same fixed-order reduction); (2) after cudaDeviceReset and fresh
 * allocations of the same inputs, the no-alloc backward (called twice)
 * reproduces the first gradients bit for bit; (3) no device error flag.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "attnres.h"

#define S_SRC 4
#define T_TOK 200
#define D_CH 7168

static uint64_t next_u64(uint64_t* x) { /* splitmix64 */
  uint64_t z = (*x += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* a finite normal bf16 bit pattern, |x| in [2^-9, 8) */
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

#define N_SRC ((size_t)S_SRC * T_TOK * D_CH)
#define N_ROW ((size_t)T_TOK * D_CH)

/* One backward on freshly allocated device copies of the inputs: the
 * no-alloc entry point (workspace == 0) or the workspace one.  Gradients
 * of the sources go to g_out (bf16 bits), of the query to gw_out. */
static int run_backward(const uint16_t* h_src, const float* h_w, const uint16_t* h_dr, int use_workspace,
                        uint16_t* g_out, float* gw_out) {
  void *d_src, *d_dr, *d_g, *d_ws = NULL;
  float *d_w, *d_gw;
  int* d_err;
  CK(cudaMalloc(&d_src, N_SRC * 2));
  CK(cudaMalloc(&d_g, N_SRC * 2));
  CK(cudaMalloc(&d_dr, N_ROW * 2));
  CK(cudaMalloc((void**)&d_w, D_CH * 4));
  CK(cudaMalloc((void**)&d_gw, D_CH * 4));
  CK(cudaMalloc((void**)&d_err, 4));
  CK(cudaMemcpy(d_src, h_src, N_SRC * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_dr, h_dr, N_ROW * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_w, h_w, D_CH * 4, cudaMemcpyHostToDevice));
  CK(cudaMemset(d_g, 0xFF, N_SRC * 2));
  CK(cudaMemset(d_err, 0, 4));
  const void* srcs[S_SRC];
  void* grads[S_SRC];
  for (int s = 0; s < S_SRC; ++s) {
    srcs[s] = (const char*)d_src + (size_t)s * N_ROW * 2;
    grads[s] = (char*)d_g + (size_t)s * N_ROW * 2;
  }
  int rc;
  if (use_workspace) {
    const int64_t ws = attnres_aggregate_backward_workspace_size(T_TOK, D_CH);
    if (ws <= 0) return 1;
    CK(cudaMalloc(&d_ws, (size_t)ws));
    rc = attnres_aggregate_backward(srcs, S_SRC, T_TOK, D_CH, ATTNRES_BF16, d_w, ATTNRES_DEFAULT_EPS, d_dr, grads, 0,
                                    d_gw, d_ws, ws, d_err, NULL);
  } else {
    rc = attnres_aggregate_backward_noalloc(srcs, S_SRC, T_TOK, D_CH, ATTNRES_BF16, d_w, ATTNRES_DEFAULT_EPS, d_dr,
                                            grads, 0, d_gw, d_err, NULL);
  }
  if (rc != ATTNRES_OK) {
    fprintf(stderr, "backward (%s): %s (%s)\n", use_workspace ? "workspace" : "no-alloc", attnres_status_string(rc),
            attnres_last_error());
    return 1;
  }
  CK(cudaDeviceSynchronize());
  int h_err = -1;
  CK(cudaMemcpy(&h_err, d_err, 4, cudaMemcpyDeviceToHost));
  if (h_err != 0) {
    fprintf(stderr, "device error flags %d\n", h_err);
    return 1;
  }
  CK(cudaMemcpy(g_out, d_g, N_SRC * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(gw_out, d_gw, D_CH * 4, cudaMemcpyDeviceToHost));
  CK(cudaFree(d_src));
  CK(cudaFree(d_g));
  CK(cudaFree(d_dr));
  CK(cudaFree(d_w));
  CK(cudaFree(d_gw));
  CK(cudaFree(d_err));
  if (d_ws) CK(cudaFree(d_ws));
  return 0;
}

int main(void) {
  uint16_t* h_src = (uint16_t*)malloc(N_SRC * 2);
  uint16_t* h_dr = (uint16_t*)malloc(N_ROW * 2);
  float* h_w = (float*)malloc(D_CH * 4);
  uint16_t* g_ref = (uint16_t*)malloc(N_SRC * 2);
  uint16_t* g_a = (uint16_t*)malloc(N_SRC * 2);
  float *gw_ref = (float*)malloc(D_CH * 4), *gw_a = (float*)malloc(D_CH * 4);
  if (!h_src || !h_dr || !h_w || !g_ref || !g_a || !gw_ref || !gw_a) return 2;
  uint64_t seed = 77123u;
  for (size_t i = 0; i < N_SRC; ++i) h_src[i] = random_bf16(&seed);
  for (size_t i = 0; i < N_ROW; ++i) h_dr[i] = random_bf16(&seed);
  for (int c = 0; c < D_CH; ++c) h_w[c] = (float)((int64_t)(next_u64(&seed) >> 40) - (1 << 23)) / (float)(1 << 23) / 42.0f;

  CK(cudaSetDevice(0));
  int rc = run_backward(h_src, h_w, h_dr, 1, g_ref, gw_ref);
  if (rc) return rc;
  rc = run_backward(h_src, h_w, h_dr, 0, g_a, gw_a);
  if (rc) return rc;
  if (memcmp(g_a, g_ref, N_SRC * 2) || memcmp(gw_a, gw_ref, D_CH * 4)) {
    fprintf(stderr, "no-alloc backward differs from the workspace backward before the reset\n");
    return 1;
  }
  for (int round = 0; round < 2; ++round) {
    if (round == 0) CK(cudaDeviceReset());
    memset(g_a, 0, N_SRC * 2);
    memset(gw_a, 0, D_CH * 4);
    rc = run_backward(h_src, h_w, h_dr, 0, g_a, gw_a);
    if (rc) return rc;
    if (memcmp(g_a, g_ref, N_SRC * 2) || memcmp(gw_a, gw_ref, D_CH * 4)) {
      fprintf(stderr, "no-alloc backward after the reset (call %d) differs from the first result\n", round + 1);
      return 1;
    }
  }
  printf("no-alloc backward: equal before and after cudaDeviceReset\n");
  return 0;
}
