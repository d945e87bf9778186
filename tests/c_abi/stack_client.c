/*
 * A plain C client of the stack calls of libattnres (include/attnres.h): no
 * Python, no torch.  It fills an attnres_state itself (the struct as C lays
 * it out, flags included) and runs a 14-layer bf16 stack with blocks of 4 --
 * attnres_layer_step, then the stand-in body attnres_synthetic_layer, per
 * layer, and the final aggregation -- twice: with flags = 0 and with
 * ATTNRES_STATE_EARLY_LOADS.  It also runs one layer through
 * attnres_aggregate_fold and through attnres_fold + attnres_aggregate.
 *
 *   stack_client OUT.bin        exit status 0 = every check passed
 *
 * Checks here: the two stack runs give the same bits (final r, every
 * layer's weights); the fused fold equals the separate calls bit for bit;
 * a state call out of order is refused with ATTNRES_ESTATE; no device error.
 * The file then lets tests/test_gpu_c_abi.py rerun the same stack through
 * the Python binding and compare bit for bit.
 *
 * File layout (little endian): int32 T, d, L, B; uint16 h0 [T][d] (bf16);
 * float32 W [L+1][d], G [L][d], Sc [L][d]; uint16 r [T][d]; float32 the
 * weights of layers 1..L+1, each [T][S_l], concatenated.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "attnres.h"

#define T_TOK 100
#define D_CH 7168
#define L_LAYERS 14
#define B_SIZE 4
#define N_BLOCKS ((L_LAYERS + B_SIZE - 1) / B_SIZE)

static uint64_t next_u64(uint64_t* x) { /* splitmix64 */
  uint64_t z = (*x += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* uniform in [-1, 1) with 24 random bits */
static float uniform_pm1(uint64_t* x) {
  return (float)((int64_t)(next_u64(x) >> 40) - (1 << 23)) / (float)(1 << 23);
}

/* bf16 bits of a finite normal number with |x| in [2^-9, 8) */
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

#define CA(call, what)                                                                              \
  do {                                                                                              \
    int rc_ = (call);                                                                               \
    if (rc_ != ATTNRES_OK) {                                                                        \
      fprintf(stderr, "%s: %s (%s)\n", what, attnres_status_string(rc_), attnres_last_error());     \
      return 1;                                                                                     \
    }                                                                                               \
  } while (0)

#define ROW ((size_t)T_TOK * D_CH)

/* device buffers of one stack run */
typedef struct {
  void *h0, *partial, *reps[N_BLOCKS], *r, *F;
  float *W, *G, *Sc, *wts;
  int* err;
} Bufs;

static int total_sources(void) {
  int n = 0;
  for (int l = 1; l <= L_LAYERS + 1; ++l) n += attnres_num_sources(l, B_SIZE, L_LAYERS);
  return n;
}

/* One stack forward with the given state flags; r and every layer's weights
 * copied back.  Ends by checking that an out-of-order step is refused. */
static int run_stack(const Bufs* b, int flags, uint16_t* r_out, float* w_out) {
  attnres_state st;
  memset(&st, 0xAB, sizeof st); /* init must set every field */
  CA(attnres_state_init(&st, b->h0, b->reps, N_BLOCKS, b->partial, T_TOK, D_CH, ATTNRES_BF16, L_LAYERS, B_SIZE,
                        ATTNRES_DEFAULT_EPS),
     "attnres_state_init");
  if (st.flags != 0 || st.folded != 0) {
    fprintf(stderr, "attnres_state_init left flags %d, folded %d\n", st.flags, st.folded);
    return 1;
  }
  st.flags = flags;
  CK(cudaMemset(b->err, 0, 4));
  size_t off = 0; /* floats of weights so far */
  for (int l = 1; l <= L_LAYERS + 1; ++l) {
    CA(attnres_layer_step(&st, l > 1 ? b->F : NULL, b->W + (size_t)(l - 1) * D_CH, l, b->r, b->wts + off, b->err,
                          NULL),
       "attnres_layer_step");
    off += (size_t)T_TOK * attnres_num_sources(l, B_SIZE, L_LAYERS);
    if (l <= L_LAYERS)
      CA(attnres_synthetic_layer(b->r, b->G + (size_t)(l - 1) * D_CH, b->Sc + (size_t)(l - 1) * D_CH, b->F, T_TOK,
                                 D_CH, ATTNRES_BF16, NULL),
         "attnres_synthetic_layer");
  }
  CK(cudaDeviceSynchronize());
  int h_err = -1;
  CK(cudaMemcpy(&h_err, b->err, 4, cudaMemcpyDeviceToHost));
  if (h_err != 0) {
    fprintf(stderr, "device error flags %d (state flags %d)\n", h_err, flags);
    return 1;
  }
  CK(cudaMemcpy(r_out, b->r, ROW * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(w_out, b->wts, off * 4, cudaMemcpyDeviceToHost));
  /* every layer is folded now: layer 3 with F_prev needs folded == 1 */
  const int rc = attnres_layer_step(&st, b->F, b->W, 3, b->r, NULL, NULL, NULL);
  if (rc != ATTNRES_ESTATE) {
    fprintf(stderr, "an out-of-order step returned %d, not ATTNRES_ESTATE\n", rc);
    return 1;
  }
  return 0;
}

/* attnres_aggregate_fold against attnres_fold + attnres_aggregate, over the
 * stack's rows as they are after a run */
static int check_fold(const Bufs* b) {
  void *dst1, *dst2, *r1, *r2;
  float *a1, *a2;
  CK(cudaMalloc(&dst1, ROW * 2));
  CK(cudaMalloc(&dst2, ROW * 2));
  CK(cudaMalloc(&r1, ROW * 2));
  CK(cudaMalloc(&r2, ROW * 2));
  CK(cudaMalloc((void**)&a1, (size_t)T_TOK * 4 * 4));
  CK(cudaMalloc((void**)&a2, (size_t)T_TOK * 4 * 4));
  const void* stored[3] = {b->h0, b->reps[0], b->reps[1]};
  CA(attnres_aggregate_fold(stored, 3, b->reps[2], b->F, dst1, T_TOK, D_CH, ATTNRES_BF16, b->W, ATTNRES_DEFAULT_EPS,
                            r1, a1, ATTNRES_STATE_EARLY_LOADS, b->err, NULL),
     "attnres_aggregate_fold");
  CA(attnres_fold(b->reps[2], b->F, dst2, T_TOK, D_CH, ATTNRES_BF16, NULL), "attnres_fold");
  const void* all[4] = {b->h0, b->reps[0], b->reps[1], dst2};
  CA(attnres_aggregate(all, 4, T_TOK, D_CH, ATTNRES_BF16, b->W, ATTNRES_DEFAULT_EPS, r2, ATTNRES_BF16, a2, b->err,
                       NULL),
     "attnres_aggregate");
  CK(cudaDeviceSynchronize());
  const size_t nb[3] = {ROW * 2, ROW * 2, (size_t)T_TOK * 4 * 4};
  void* x[3] = {dst1, r1, a1};
  void* y[3] = {dst2, r2, a2};
  for (int k = 0; k < 3; ++k) {
    unsigned char* hx = (unsigned char*)malloc(nb[k]);
    unsigned char* hy = (unsigned char*)malloc(nb[k]);
    if (!hx || !hy) return 2;
    CK(cudaMemcpy(hx, x[k], nb[k], cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(hy, y[k], nb[k], cudaMemcpyDeviceToHost));
    const int same = memcmp(hx, hy, nb[k]) == 0;
    free(hx);
    free(hy);
    if (!same) {
      fprintf(stderr, "attnres_aggregate_fold differs from fold + aggregate (output %d)\n", k);
      return 1;
    }
  }
  CK(cudaFree(dst1));
  CK(cudaFree(dst2));
  CK(cudaFree(r1));
  CK(cudaFree(r2));
  CK(cudaFree(a1));
  CK(cudaFree(a2));
  return 0;
}

int main(int argc, char** argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s OUT.bin\n", argv[0]);
    return 2;
  }
  const int nw = total_sources() * T_TOK; /* floats of weights, all layers */
  uint16_t* h_h0 = (uint16_t*)malloc(ROW * 2);
  float* h_W = (float*)malloc((size_t)(L_LAYERS + 1) * D_CH * 4);
  float* h_G = (float*)malloc((size_t)L_LAYERS * D_CH * 4);
  float* h_Sc = (float*)malloc((size_t)L_LAYERS * D_CH * 4);
  uint16_t *h_r0 = (uint16_t*)malloc(ROW * 2), *h_r1 = (uint16_t*)malloc(ROW * 2);
  float *h_w0 = (float*)malloc((size_t)nw * 4), *h_w1 = (float*)malloc((size_t)nw * 4);
  if (!h_h0 || !h_W || !h_G || !h_Sc || !h_r0 || !h_r1 || !h_w0 || !h_w1) return 2;
  uint64_t seed = 5150u;
  for (size_t i = 0; i < ROW; ++i) h_h0[i] = random_bf16(&seed);
  for (size_t i = 0; i < (size_t)(L_LAYERS + 1) * D_CH; ++i) h_W[i] = uniform_pm1(&seed) / 42.0f;
  for (size_t i = 0; i < (size_t)L_LAYERS * D_CH; ++i) h_G[i] = 2.0f * uniform_pm1(&seed);
  for (size_t i = 0; i < (size_t)L_LAYERS * D_CH; ++i) h_Sc[i] = 0.125f + 0.075f * uniform_pm1(&seed);

  CK(cudaSetDevice(0));
  Bufs b;
  CK(cudaMalloc(&b.h0, ROW * 2));
  CK(cudaMalloc(&b.partial, ROW * 2));
  for (int k = 0; k < N_BLOCKS; ++k) CK(cudaMalloc(&b.reps[k], ROW * 2));
  CK(cudaMalloc(&b.r, ROW * 2));
  CK(cudaMalloc(&b.F, ROW * 2));
  CK(cudaMalloc((void**)&b.W, (size_t)(L_LAYERS + 1) * D_CH * 4));
  CK(cudaMalloc((void**)&b.G, (size_t)L_LAYERS * D_CH * 4));
  CK(cudaMalloc((void**)&b.Sc, (size_t)L_LAYERS * D_CH * 4));
  CK(cudaMalloc((void**)&b.wts, (size_t)nw * 4));
  CK(cudaMalloc((void**)&b.err, 4));
  CK(cudaMemcpy(b.h0, h_h0, ROW * 2, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(b.W, h_W, (size_t)(L_LAYERS + 1) * D_CH * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(b.G, h_G, (size_t)L_LAYERS * D_CH * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(b.Sc, h_Sc, (size_t)L_LAYERS * D_CH * 4, cudaMemcpyHostToDevice));

  int rc = run_stack(&b, 0, h_r0, h_w0);
  if (rc) return rc;
  rc = run_stack(&b, ATTNRES_STATE_EARLY_LOADS, h_r1, h_w1);
  if (rc) return rc;
  if (memcmp(h_r0, h_r1, ROW * 2) || memcmp(h_w0, h_w1, (size_t)nw * 4)) {
    fprintf(stderr, "the stack with early loads differs from the stack without\n");
    return 1;
  }
  rc = check_fold(&b);
  if (rc) return rc;

  FILE* f = fopen(argv[1], "wb");
  if (!f) return 2;
  const int32_t hdr[4] = {T_TOK, D_CH, L_LAYERS, B_SIZE};
  fwrite(hdr, 4, 4, f);
  fwrite(h_h0, 2, ROW, f);
  fwrite(h_W, 4, (size_t)(L_LAYERS + 1) * D_CH, f);
  fwrite(h_G, 4, (size_t)L_LAYERS * D_CH, f);
  fwrite(h_Sc, 4, (size_t)L_LAYERS * D_CH, f);
  fwrite(h_r1, 2, ROW, f);
  fwrite(h_w1, 4, (size_t)nw, f);
  fclose(f);
  printf("stack client: early loads = plain bit for bit; aggregate_fold = fold + aggregate\n");
  return 0;
}
