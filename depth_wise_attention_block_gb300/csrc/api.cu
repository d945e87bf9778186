// The C ABI of libattnres (declared in include/attnres.h): argument
// checking, the host-side block bookkeeping of a stack (which sources layer
// l reads, where the folded layer output goes), and dispatch to the kernels.
//
// Block bookkeeping follows the Kimi K3 chaptered tutorial (kimi.papertok.ai),
// ch. 4.3 Eq. 10 (two-case value list; no source for an empty partial sum;
// the final output layer aggregates all block representations) and ch. 4.5
// (an incomplete last block).
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cmath>
#include <string>

#include "attnres.h"
#include "launch.h"

using namespace attnres;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return ATTNRES_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTNRES_ECUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool valid_dtype(int dt) { return dt == ATTNRES_F32 || dt == ATTNRES_BF16; }

// Whether the byte ranges [a, a + na) and [b, b + nb) share a byte.
bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && pa < pb + (uintptr_t)nb && pb < pa + (uintptr_t)na;
}

// The output r (and the weights) must not share memory with any source.
int check_outputs_apart(const void* const* sources, int S, int64_t src_bytes, const void* out_r, int64_t r_bytes,
                        const void* out_a, int64_t a_bytes) {
  for (int s = 0; s < S; ++s) {
    if (overlaps(out_r, r_bytes, sources[s], src_bytes)) return fail(ATTNRES_EINVAL, "r overlaps source %d", s);
    if (out_a && overlaps(out_a, a_bytes, sources[s], src_bytes))
      return fail(ATTNRES_EINVAL, "the weights overlap source %d", s);
  }
  if (out_a && overlaps(out_a, a_bytes, out_r, r_bytes)) return fail(ATTNRES_EINVAL, "the weights overlap r");
  return ATTNRES_OK;
}

// Each source gradient must share no byte with a source, with grad_r or
// with another gradient (row = bytes of one [T, d] row).
int check_grads_apart(const void* const* sources, void* const* grads, int S, int64_t row, const void* grad_r) {
  for (int s = 0; s < S; ++s) {
    for (int j = 0; j < S; ++j)
      if (overlaps(grads[s], row, sources[j], row))
        return fail(ATTNRES_EINVAL, "grad_sources[%d] overlaps sources[%d]", s, j);
    for (int j = 0; j < s; ++j)
      if (overlaps(grads[s], row, grads[j], row))
        return fail(ATTNRES_EINVAL, "grad_sources[%d] overlaps grad_sources[%d]", s, j);
    if (overlaps(grads[s], row, grad_r, row)) return fail(ATTNRES_EINVAL, "grad_sources[%d] overlaps grad_r", s);
  }
  return ATTNRES_OK;
}

// T * d * 4 must stay well inside int64 (element offsets are 64-bit).
bool size_ok(int64_t T, int d) { return T >= 0 && d >= 1 && T <= (((int64_t)1) << 40) / d; }

int num_blocks(int L, int B) { return (L + B - 1) / B; }

// Where folding layer p's output goes, and what the partial sum held before.
struct FoldPlan {
  int block;        // n: block of layer p (1-based)
  bool has_prev;    // partial sum non-empty before folding v_p
  bool ends_block;  // p is the last layer of block n
};

FoldPlan fold_plan(int p, int B, int L) {
  FoldPlan f;
  f.block = (p - 1) / B + 1;
  const int first = (f.block - 1) * B + 1;
  f.has_prev = p > first;
  f.ends_block = (p % B == 0) || (p == L);
  return f;
}

// Sources of layer folded + 1 of a state with every earlier layer output
// folded: [h_0, b_1 .. b_c, partial (if open)] (Eq. 10).  Returns S.
int state_sources(const attnres_state* st, const void** out) {
  int S = 0;
  out[S++] = st->h0;
  const int f = st->folded;
  int completed = 0;
  bool partial = false;
  if (f > 0) {
    const FoldPlan fp = fold_plan(f, st->block_size, st->num_layers);
    completed = fp.ends_block ? fp.block : fp.block - 1;
    partial = !fp.ends_block;
  }
  for (int k = 0; k < completed; ++k) out[S++] = st->block_reps[k];
  if (partial) out[S++] = st->partial;
  return S;
}

int check_state(const attnres_state* st) {
  if (!st) return fail(ATTNRES_EINVAL, "state is NULL");
  if (!st->h0 || !st->partial) return fail(ATTNRES_EINVAL, "state h0/partial is NULL");
  if (!valid_dtype(st->dtype)) return fail(ATTNRES_EDTYPE, "state dtype %d", st->dtype);
  if (!size_ok(st->T, st->d)) return fail(ATTNRES_EINVAL, "state T=%lld d=%d", (long long)st->T, st->d);
  if (st->num_layers < 1 || st->block_size < 1) return fail(ATTNRES_EINVAL, "state L/B");
  if (num_blocks(st->num_layers, st->block_size) > ATTNRES_MAX_BLOCKS) return fail(ATTNRES_ERANGE, "too many blocks");
  if (st->folded < 0 || st->folded > st->num_layers) return fail(ATTNRES_ESTATE, "state folded=%d", st->folded);
  return ATTNRES_OK;
}


// ---- host-buffer aggregation: staging-slot layout and the copy pipeline ----

constexpr int kMaxHostSlots = 8;  // more than 3 slots gains nothing; bounds the events made per call

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }
int64_t dtype_bytes(int dt) { return dt == ATTNRES_BF16 ? 2 : 4; }

// Workspace: the query (d fp32), then per slot the [S, n, d] sources of a
// chunk of n <= chunk_tokens tokens, its r and (optionally) its weights.
struct HostLayout {
  int64_t w_bytes, src_bytes, r_bytes, a_bytes, slot_bytes;
};

HostLayout host_layout(int S, int64_t Tc, int d, int src_dtype, int out_dtype, bool with_weights) {
  HostLayout L;
  L.w_bytes = align256(int64_t(d) * 4);
  L.src_bytes = align256(int64_t(S) * Tc * d * dtype_bytes(src_dtype));
  L.r_bytes = align256(Tc * d * dtype_bytes(out_dtype));
  L.a_bytes = with_weights ? align256(Tc * S * 4) : 0;
  L.slot_bytes = L.src_bytes + L.r_bytes + L.a_bytes;
  return L;
}

// The two copy streams and the per-slot events of one call; released when
// the call returns (CUDA defers the release until queued work is done).
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t arrived[kMaxHostSlots] = {}, computed[kMaxHostSlots] = {}, drained[kMaxHostSlots] = {};

  cudaError_t create(int nslots) {
    cudaError_t e = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming);
    for (int k = 0; k < nslots && e == cudaSuccess; ++k) {
      e = cudaEventCreateWithFlags(&arrived[k], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&computed[k], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&drained[k], cudaEventDisableTiming);
    }
    return e;
  }

  ~HostPipe() {
    for (int k = 0; k < kMaxHostSlots; ++k) {
      if (arrived[k]) cudaEventDestroy(arrived[k]);
      if (computed[k]) cudaEventDestroy(computed[k]);
      if (drained[k]) cudaEventDestroy(drained[k]);
    }
    if (start) cudaEventDestroy(start);
    if (in) cudaStreamDestroy(in);
    if (out) cudaStreamDestroy(out);
  }
};

}  // namespace

extern "C" {

int attnres_version(void) { return (2 << 16) | 0; }

const char* attnres_status_string(int status) {
  switch (status) {
    case ATTNRES_OK: return "ATTNRES_OK";
    case ATTNRES_EINVAL: return "ATTNRES_EINVAL: invalid argument";
    case ATTNRES_EDTYPE: return "ATTNRES_EDTYPE: unsupported dtype";
    case ATTNRES_ERANGE: return "ATTNRES_ERANGE: size out of range";
    case ATTNRES_ECUDA: return "ATTNRES_ECUDA: CUDA error";
    case ATTNRES_ESTATE: return "ATTNRES_ESTATE: stack call out of order";
    default: return "unknown attnres status";
  }
}

const char* attnres_last_error(void) { return g_last_error.c_str(); }

int attnres_aggregate(const void* const* sources, int S, int64_t T, int d, int src_dtype, const float* w_l, float eps,
                      void* out_r, int out_dtype, float* out_weights, int* dev_err, void* stream) {
  if (!sources) return fail(ATTNRES_EINVAL, "sources is NULL");
  if (S < 1) return fail(ATTNRES_EINVAL, "S=%d < 1", S);
  if (S > ATTNRES_MAX_SOURCES) return fail(ATTNRES_ERANGE, "S=%d > %d", S, ATTNRES_MAX_SOURCES);
  if (!valid_dtype(src_dtype) || !valid_dtype(out_dtype)) return fail(ATTNRES_EDTYPE, "dtype %d/%d", src_dtype, out_dtype);
  if (T < 0 || d < 1) return fail(ATTNRES_EINVAL, "T=%lld d=%d", (long long)T, d);
  if (!size_ok(T, d)) return fail(ATTNRES_ERANGE, "T*d too large");
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(ATTNRES_EINVAL, "eps must be finite and >= 0");
  if (T == 0) return ok();  // empty problem: nothing is read or written, buffers may be NULL
  if (!w_l || !out_r) return fail(ATTNRES_EINVAL, "w_l/out_r is NULL");
  for (int s = 0; s < S; ++s)
    if (!sources[s]) return fail(ATTNRES_EINVAL, "sources[%d] is NULL", s);
  {
    const int64_t isz = src_dtype == ATTNRES_BF16 ? 2 : 4, osz = out_dtype == ATTNRES_BF16 ? 2 : 4;
    const int rc = check_outputs_apart(sources, S, T * d * isz, out_r, T * d * osz, out_weights, T * S * 4);
    if (rc != ATTNRES_OK) return rc;
  }
  AggArgs a{};
  for (int s = 0; s < S; ++s) a.src[s] = sources[s];
  a.n_stored = S;
  a.T = T;
  a.d = d;
  a.src_dtype = src_dtype;
  a.w = w_l;
  a.eps = eps;
  a.out_r = out_r;
  a.out_dtype = out_dtype;
  a.out_a = out_weights;
  a.dev_err = dev_err;
  a.stream = static_cast<cudaStream_t>(stream);
  AggPath path;
  cudaError_t e = launch_aggregate(a, &path);
  if (e != cudaSuccess) return cuda_fail(e, "attnres_aggregate launch");
  return ok();
}

int attnres_aggregate_fold(const void* const* sources, int n_stored, const void* prev, const void* F, void* dst,
                           int64_t T, int d, int dtype, const float* w_l, float eps, void* out_r,
                           float* out_weights, int flags, int* dev_err, void* stream) {
  if (n_stored < 0) return fail(ATTNRES_EINVAL, "n_stored=%d < 0", n_stored);
  if (n_stored + 1 > ATTNRES_MAX_SOURCES) return fail(ATTNRES_ERANGE, "S=%d > %d", n_stored + 1, ATTNRES_MAX_SOURCES);
  if (n_stored > 0 && !sources) return fail(ATTNRES_EINVAL, "sources is NULL");
  if (!valid_dtype(dtype)) return fail(ATTNRES_EDTYPE, "dtype %d", dtype);
  if (T < 0 || d < 1) return fail(ATTNRES_EINVAL, "T=%lld d=%d", (long long)T, d);
  if (!size_ok(T, d)) return fail(ATTNRES_ERANGE, "T*d too large");
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(ATTNRES_EINVAL, "eps must be finite and >= 0");
  if (flags & ~ATTNRES_STATE_EARLY_LOADS) return fail(ATTNRES_EINVAL, "flags 0x%x: unknown bits", flags);
  if (T == 0) return ok();
  if (!w_l || !out_r || !F || !dst) return fail(ATTNRES_EINVAL, "w_l/out_r/F/dst is NULL");
  for (int s = 0; s < n_stored; ++s)
    if (!sources[s]) return fail(ATTNRES_EINVAL, "sources[%d] is NULL", s);
  {
    const int S = n_stored + 1;
    const int64_t row = T * d * (dtype == ATTNRES_BF16 ? 2 : 4);
    // every row read: the stored sources, prev, F, and dst (the new source)
    const void* rows[ATTNRES_MAX_SOURCES + 2];
    int nr = 0;
    for (int s = 0; s < n_stored; ++s) rows[nr++] = sources[s];
    if (prev) rows[nr++] = prev;
    rows[nr++] = F;
    rows[nr++] = dst;
    const int rc = check_outputs_apart(rows, nr, row, out_r, row, out_weights, T * S * 4);
    if (rc != ATTNRES_OK) return rc;
    // dst is written while the rows are read: apart from all of them, except
    // that it may be prev itself (the partial sum updated in place)
    for (int s = 0; s < n_stored; ++s)
      if (overlaps(dst, row, sources[s], row)) return fail(ATTNRES_EINVAL, "dst overlaps sources[%d]", s);
    if (overlaps(dst, row, F, row)) return fail(ATTNRES_EINVAL, "dst overlaps F");
    if (prev && prev != dst && overlaps(dst, row, prev, row))
      return fail(ATTNRES_EINVAL, "dst overlaps prev without being prev");
  }
  AggArgs a{};
  for (int s = 0; s < n_stored; ++s) a.src[s] = sources[s];
  a.n_stored = n_stored;
  a.fuse_prev = prev;
  a.fuse_F = F;
  a.fuse_dst = dst;
  a.early_loads = (flags & ATTNRES_STATE_EARLY_LOADS) != 0;
  a.T = T;
  a.d = d;
  a.src_dtype = dtype;
  a.w = w_l;
  a.eps = eps;
  a.out_r = out_r;
  a.out_dtype = dtype;
  a.out_a = out_weights;
  a.dev_err = dev_err;
  a.stream = static_cast<cudaStream_t>(stream);
  AggPath path;
  cudaError_t e = launch_aggregate(a, &path);
  if (e != cudaSuccess) return cuda_fail(e, "attnres_aggregate_fold launch");
  return ok();
}

int64_t attnres_aggregate_host_workspace_size(int S, int64_t chunk_tokens, int d, int src_dtype, int out_dtype,
                                              int with_weights, int slots) {
  if (S < 1) return fail(ATTNRES_EINVAL, "S=%d < 1", S);
  if (S > ATTNRES_MAX_SOURCES) return fail(ATTNRES_ERANGE, "S=%d > %d", S, ATTNRES_MAX_SOURCES);
  if (!valid_dtype(src_dtype) || !valid_dtype(out_dtype)) return fail(ATTNRES_EDTYPE, "dtype %d/%d", src_dtype, out_dtype);
  if (chunk_tokens < 1 || d < 1) return fail(ATTNRES_EINVAL, "chunk_tokens=%lld d=%d", (long long)chunk_tokens, d);
  if (!size_ok(chunk_tokens, d)) return fail(ATTNRES_ERANGE, "chunk_tokens*d too large");
  if (with_weights != 0 && with_weights != 1) return fail(ATTNRES_EINVAL, "with_weights must be 0 or 1");
  if (slots < 1 || slots > kMaxHostSlots) return fail(ATTNRES_EINVAL, "slots=%d not in 1..%d", slots, kMaxHostSlots);
  const HostLayout L = host_layout(S, chunk_tokens, d, src_dtype, out_dtype, with_weights != 0);
  ok();
  return L.w_bytes + int64_t(slots) * L.slot_bytes;
}

int attnres_aggregate_host(const void* const* sources_host, int S, int64_t T, int d, int src_dtype,
                           const float* w_host, float eps, void* r_host, int out_dtype, float* weights_host,
                           int64_t chunk_tokens, void* workspace, int64_t workspace_bytes, int* dev_err,
                           void* stream) {
  if (!sources_host) return fail(ATTNRES_EINVAL, "sources_host is NULL");
  if (S < 1) return fail(ATTNRES_EINVAL, "S=%d < 1", S);
  if (S > ATTNRES_MAX_SOURCES) return fail(ATTNRES_ERANGE, "S=%d > %d", S, ATTNRES_MAX_SOURCES);
  if (!valid_dtype(src_dtype) || !valid_dtype(out_dtype)) return fail(ATTNRES_EDTYPE, "dtype %d/%d", src_dtype, out_dtype);
  if (T < 0 || d < 1) return fail(ATTNRES_EINVAL, "T=%lld d=%d", (long long)T, d);
  if (!size_ok(T, d)) return fail(ATTNRES_ERANGE, "T*d too large");
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(ATTNRES_EINVAL, "eps must be finite and >= 0");
  if (chunk_tokens < 1) return fail(ATTNRES_EINVAL, "chunk_tokens=%lld < 1", (long long)chunk_tokens);
  if (T == 0) return ok();
  if (!w_host || !r_host || !workspace) return fail(ATTNRES_EINVAL, "w_host/r_host/workspace is NULL");
  for (int s = 0; s < S; ++s)
    if (!sources_host[s]) return fail(ATTNRES_EINVAL, "sources_host[%d] is NULL", s);
  {
    const int64_t isz = src_dtype == ATTNRES_BF16 ? 2 : 4, osz = out_dtype == ATTNRES_BF16 ? 2 : 4;
    const int rc = check_outputs_apart(sources_host, S, T * d * isz, r_host, T * d * osz, weights_host, T * S * 4);
    if (rc != ATTNRES_OK) return rc;
  }
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return fail(ATTNRES_EINVAL, "workspace not 256-byte aligned");
  const int64_t Tc = chunk_tokens < T ? chunk_tokens : T;
  const int64_t nchunks = (T + Tc - 1) / Tc;
  const HostLayout L = host_layout(S, Tc, d, src_dtype, out_dtype, weights_host != nullptr);
  if (workspace_bytes < L.w_bytes + L.slot_bytes)
    return fail(ATTNRES_ERANGE, "workspace %lld bytes < %lld needed for one slot of %lld tokens",
                (long long)workspace_bytes, (long long)(L.w_bytes + L.slot_bytes), (long long)Tc);
  int64_t fit = (workspace_bytes - L.w_bytes) / L.slot_bytes;
  if (fit > nchunks) fit = nchunks;
  const int nslots = fit > kMaxHostSlots ? kMaxHostSlots : int(fit);

  const int64_t es = dtype_bytes(src_dtype), os = dtype_bytes(out_dtype);
  cudaStream_t user = static_cast<cudaStream_t>(stream);
  // Copies on streams of its own cannot join a capture: refuse it up front
  // rather than invalidate the caller's capture half way.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t ce = cudaStreamIsCapturing(user, &cap);
  if (ce != cudaSuccess) return cuda_fail(ce, "attnres_aggregate_host: cudaStreamIsCapturing");
  if (cap != cudaStreamCaptureStatusNone) return fail(ATTNRES_EINVAL, "stream is being captured into a graph");
  HostPipe pipe;
  cudaError_t e = pipe.create(nslots);
  if (e != cudaSuccess) return cuda_fail(e, "attnres_aggregate_host: creating copy streams/events");
  // On a failure part way, work issued on `stream` afterwards must still
  // wait for every copy already queued (the caller may free the buffers
  // once it has synchronised): join both copy streams, best effort.
  auto join_copies = [&]() {
    if (cudaEventRecord(pipe.start, pipe.in) == cudaSuccess) cudaStreamWaitEvent(user, pipe.start, 0);
    if (cudaEventRecord(pipe.arrived[0], pipe.out) == cudaSuccess) cudaStreamWaitEvent(user, pipe.arrived[0], 0);
  };
#define HOST_CK(call)                                           \
  do {                                                          \
    cudaError_t e_ = (call);                                    \
    if (e_ != cudaSuccess) {                                    \
      const int rc_ = cuda_fail(e_, "attnres_aggregate_host: " #call); \
      join_copies();                                            \
      return rc_;                                               \
    }                                                           \
  } while (0)

  char* ws = static_cast<char*>(workspace);
  float* w_dev = reinterpret_cast<float*>(ws);
  HOST_CK(cudaEventRecord(pipe.start, user));  // after the work already on `stream`
  HOST_CK(cudaStreamWaitEvent(pipe.in, pipe.start, 0));
  HOST_CK(cudaMemcpyAsync(w_dev, w_host, size_t(d) * 4, cudaMemcpyHostToDevice, pipe.in));
  for (int64_t c = 0; c < nchunks; ++c) {
    const int k = int(c % nslots);
    const int64_t t0 = c * Tc, n = (T - t0) < Tc ? (T - t0) : Tc;
    char* slot = ws + L.w_bytes + int64_t(k) * L.slot_bytes;
    char* r_dev = slot + L.src_bytes;
    float* a_dev = weights_host ? reinterpret_cast<float*>(slot + L.src_bytes + L.r_bytes) : nullptr;
    // The slot is free again once the chunk that used it last has been copied out.
    if (c >= nslots) HOST_CK(cudaStreamWaitEvent(pipe.in, pipe.drained[k], 0));
    AggArgs a{};
    for (int s = 0; s < S; ++s) {
      char* dst = slot + int64_t(s) * n * d * es;  // [S, n, d] in the slot
      HOST_CK(cudaMemcpyAsync(dst, static_cast<const char*>(sources_host[s]) + t0 * d * es, size_t(n * d * es),
                              cudaMemcpyHostToDevice, pipe.in));
      a.src[s] = dst;
    }
    HOST_CK(cudaEventRecord(pipe.arrived[k], pipe.in));
    HOST_CK(cudaStreamWaitEvent(user, pipe.arrived[k], 0));
    a.n_stored = S;
    a.T = n;
    a.d = d;
    a.src_dtype = src_dtype;
    a.w = w_dev;
    a.eps = eps;
    a.out_r = r_dev;
    a.out_dtype = out_dtype;
    a.out_a = a_dev;
    a.dev_err = dev_err;
    a.stream = user;
    AggPath path;
    HOST_CK(launch_aggregate(a, &path));
    HOST_CK(cudaEventRecord(pipe.computed[k], user));
    HOST_CK(cudaStreamWaitEvent(pipe.out, pipe.computed[k], 0));
    HOST_CK(cudaMemcpyAsync(static_cast<char*>(r_host) + t0 * d * os, r_dev, size_t(n * d * os),
                            cudaMemcpyDeviceToHost, pipe.out));
    if (weights_host)
      HOST_CK(cudaMemcpyAsync(weights_host + t0 * S, a_dev, size_t(n * S * 4), cudaMemcpyDeviceToHost, pipe.out));
    HOST_CK(cudaEventRecord(pipe.drained[k], pipe.out));
  }
  // The copy-out stream is in order: its last event covers every chunk.
  HOST_CK(cudaStreamWaitEvent(user, pipe.drained[(nchunks - 1) % nslots], 0));
#undef HOST_CK
  return ok();
}

int64_t attnres_aggregate_backward_workspace_size(int64_t T, int d) {
  if (T < 0 || d < 1) return fail(ATTNRES_EINVAL, "T=%lld d=%d", (long long)T, d);
  if (!size_ok(T, d)) return fail(ATTNRES_ERANGE, "T*d too large");
  const int64_t nb = backward_blocks(T);
  if (nb < 0) return fail(ATTNRES_ECUDA, "no CUDA device");
  ok();
  return nb * (int64_t)d * (int64_t)sizeof(float);
}

int attnres_aggregate_backward(const void* const* sources, int S, int64_t T, int d, int dtype, const float* w_l,
                               float eps, const void* grad_r, void* const* grad_sources, int accumulate,
                               float* grad_w, void* workspace, int64_t workspace_bytes, int* dev_err, void* stream) {
  if (!sources || !grad_sources) return fail(ATTNRES_EINVAL, "sources/grad_sources is NULL");
  if (S < 1) return fail(ATTNRES_EINVAL, "S=%d < 1", S);
  if (S > ATTNRES_MAX_SOURCES) return fail(ATTNRES_ERANGE, "S=%d > %d", S, ATTNRES_MAX_SOURCES);
  if (!valid_dtype(dtype)) return fail(ATTNRES_EDTYPE, "dtype %d", dtype);
  if (T < 0 || d < 1) return fail(ATTNRES_EINVAL, "T=%lld d=%d", (long long)T, d);
  if (!size_ok(T, d)) return fail(ATTNRES_ERANGE, "T*d too large");
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(ATTNRES_EINVAL, "eps must be finite and >= 0");
  if (!grad_w) return fail(ATTNRES_EINVAL, "grad_w is NULL");
  if (accumulate != 0 && accumulate != 1) return fail(ATTNRES_EINVAL, "accumulate must be 0 or 1");
  if (T > 0) {
    if (!w_l || !grad_r || !workspace) return fail(ATTNRES_EINVAL, "w_l/grad_r/workspace is NULL");
    for (int s = 0; s < S; ++s) {
      if (!sources[s] || !grad_sources[s]) return fail(ATTNRES_EINVAL, "sources[%d]/grad_sources[%d] is NULL", s, s);
    }
    {
      const int rc = check_grads_apart(sources, grad_sources, S, T * d * (dtype == ATTNRES_BF16 ? 2 : 4), grad_r);
      if (rc != ATTNRES_OK) return rc;
    }
    if ((reinterpret_cast<uintptr_t>(workspace) & 3u) != 0) return fail(ATTNRES_EINVAL, "workspace not 4-byte aligned");
    const int64_t need = attnres_aggregate_backward_workspace_size(T, d);
    if (need < 0) return (int)need;
    if (workspace_bytes < need)
      return fail(ATTNRES_ERANGE, "workspace %lld bytes < %lld needed", (long long)workspace_bytes, (long long)need);
  }
  BwdArgs a{};
  for (int s = 0; s < S && T > 0; ++s) {
    a.src[s] = sources[s];
    a.grad_src[s] = grad_sources[s];
  }
  a.S = S;
  a.T = T;
  a.d = d;
  a.dtype = dtype;
  a.w = w_l;
  a.eps = eps;
  a.grad_r = grad_r;
  a.accumulate = accumulate != 0;
  a.grad_w = grad_w;
  a.workspace = static_cast<float*>(workspace);
  a.dev_err = dev_err;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_aggregate_backward(a);
  if (e != cudaSuccess) return cuda_fail(e, "attnres_aggregate_backward launch");
  return ok();
}

int attnres_aggregate_backward_noalloc(const void* const* sources, int S, int64_t T, int d, int dtype,
                                       const float* w_l, float eps, const void* grad_r, void* const* grad_sources,
                                       int accumulate, float* grad_w, int* dev_err, void* stream) {
  if (!sources || !grad_sources) return fail(ATTNRES_EINVAL, "sources/grad_sources is NULL");
  if (S < 1) return fail(ATTNRES_EINVAL, "S=%d < 1", S);
  if (S > ATTNRES_MAX_SOURCES) return fail(ATTNRES_ERANGE, "S=%d > %d", S, ATTNRES_MAX_SOURCES);
  if (!valid_dtype(dtype)) return fail(ATTNRES_EDTYPE, "dtype %d", dtype);
  if (T < 0 || d < 1) return fail(ATTNRES_EINVAL, "T=%lld d=%d", (long long)T, d);
  if (!size_ok(T, d)) return fail(ATTNRES_ERANGE, "T*d too large");
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(ATTNRES_EINVAL, "eps must be finite and >= 0");
  if (!grad_w) return fail(ATTNRES_EINVAL, "grad_w is NULL");
  if (accumulate != 0 && accumulate != 1) return fail(ATTNRES_EINVAL, "accumulate must be 0 or 1");
  float* scratch = nullptr;
  int64_t capacity = 0;
  if (T > 0) {
    if (!w_l || !grad_r) return fail(ATTNRES_EINVAL, "w_l/grad_r is NULL");
    for (int s = 0; s < S; ++s) {
      if (!sources[s] || !grad_sources[s]) return fail(ATTNRES_EINVAL, "sources[%d]/grad_sources[%d] is NULL", s, s);
    }
    {
      const int rc = check_grads_apart(sources, grad_sources, S, T * d * (dtype == ATTNRES_BF16 ? 2 : 4), grad_r);
      if (rc != ATTNRES_OK) return rc;
    }
    const int64_t rows = backward_blocks(T);
    if (rows < 0) return fail(ATTNRES_ECUDA, "no CUDA device");
    cudaError_t e = noalloc_backward_scratch(&scratch, &capacity);
    if (e != cudaSuccess) return cuda_fail(e, "attnres_aggregate_backward_noalloc scratch lookup");
    if (rows * (int64_t)d > capacity)
      return fail(ATTNRES_ERANGE,
                  "attnres_aggregate_backward_noalloc: needs %lld fp32 scratch values (%lld rows x d=%d), the "
                  "built-in scratch holds %lld; use attnres_aggregate_backward with a workspace",
                  (long long)(rows * (int64_t)d), (long long)rows, d, (long long)capacity);
  }
  BwdArgs a{};
  for (int s = 0; s < S && T > 0; ++s) {
    a.src[s] = sources[s];
    a.grad_src[s] = grad_sources[s];
  }
  a.S = S;
  a.T = T;
  a.d = d;
  a.dtype = dtype;
  a.w = w_l;
  a.eps = eps;
  a.grad_r = grad_r;
  a.accumulate = accumulate != 0;
  a.grad_w = grad_w;
  a.workspace = scratch;
  a.dev_err = dev_err;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_aggregate_backward(a);
  if (e != cudaSuccess) return cuda_fail(e, "attnres_aggregate_backward_noalloc launch");
  return ok();
}

int64_t attnres_interblock_workspace_size(int n, int64_t T, int d, int dtype, int Q) {
  if (n < 1 || n > 9) return fail(ATTNRES_ERANGE, "n=%d cached sources: 1..9", n);
  if (Q < 1 || Q > kMaxQueries) return fail(ATTNRES_ERANGE, "Q=%d queries: 1..%d", Q, kMaxQueries);
  if (!valid_dtype(dtype)) return fail(ATTNRES_EDTYPE, "dtype %d", dtype);
  if (T < 0 || d < 1 || !size_ok(T, d)) return fail(ATTNRES_EINVAL, "T=%lld d=%d", (long long)T, d);
  const int64_t b = interblock_tc_workspace_bytes(n, T, d, dtype, Q);
  if (b < 0) return fail(ATTNRES_ECUDA, "no CUDA device");
  ok();
  return b;
}

int attnres_interblock(const void* const* sources, int n, int64_t T, int d, int dtype,
                       const float* const* w_queries, int Q, float eps, float* out_r, float* out_lse,
                       float* out_weights, void* out_r0, float* out_weights0, void* workspace,
                       int64_t workspace_bytes, int* dev_err, void* stream) {
  if (!sources || !w_queries) return fail(ATTNRES_EINVAL, "sources/w_queries is NULL");
  if (n < 1 || n > 9) return fail(ATTNRES_ERANGE, "n=%d cached sources: 1..9", n);
  if (Q < 1 || Q > kMaxQueries) return fail(ATTNRES_ERANGE, "Q=%d queries: 1..%d", Q, kMaxQueries);
  if (!valid_dtype(dtype)) return fail(ATTNRES_EDTYPE, "dtype %d", dtype);
  if (T < 0 || d < 1) return fail(ATTNRES_EINVAL, "T=%lld d=%d", (long long)T, d);
  if (!size_ok(T, d)) return fail(ATTNRES_ERANGE, "T*d too large");
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(ATTNRES_EINVAL, "eps must be finite and >= 0");
  if (!twophase_supported(d, dtype))
    return fail(ATTNRES_ERANGE, "two-phase schedule needs rows of a 16-byte multiple, at most 2 x 448 vectors");
  if (T == 0) return ok();
  if (!out_r || !out_lse) return fail(ATTNRES_EINVAL, "out_r/out_lse is NULL");
  InterArgs a{};
  for (int s = 0; s < n; ++s) {
    if (!sources[s]) return fail(ATTNRES_EINVAL, "sources[%d] is NULL", s);
    if (!twophase_pointers_ok(sources[s])) return fail(ATTNRES_EINVAL, "sources[%d] not 16-byte aligned", s);
    a.src[s] = sources[s];
  }
  for (int q = 0; q < Q; ++q) {
    if (!w_queries[q]) return fail(ATTNRES_EINVAL, "w_queries[%d] is NULL", q);
    if (!twophase_pointers_ok(w_queries[q])) return fail(ATTNRES_EINVAL, "w_queries[%d] not 16-byte aligned", q);
    a.wq[q] = w_queries[q];
  }
  {
    // the outputs ([Q, T, d] fp32 r, [Q, T] lse, [Q, T, n] weights) must not
    // share memory with a source or with each other
    const int64_t row = T * d * (dtype == ATTNRES_BF16 ? 2 : 4);
    const int64_t r_bytes = (int64_t)Q * T * d * 4, lse_bytes = (int64_t)Q * T * 4, a_bytes = (int64_t)Q * T * n * 4;
    const int rc = check_outputs_apart(sources, n, row, out_r, r_bytes, out_weights, a_bytes);
    if (rc != ATTNRES_OK) return rc;
    for (int s = 0; s < n; ++s)
      if (overlaps(out_lse, lse_bytes, sources[s], row)) return fail(ATTNRES_EINVAL, "out_lse overlaps source %d", s);
    if (overlaps(out_lse, lse_bytes, out_r, r_bytes) || (out_weights && overlaps(out_lse, lse_bytes, out_weights, a_bytes)))
      return fail(ATTNRES_EINVAL, "out_lse overlaps another output");
    // the block's first-layer outputs: apart from the sources and every other output
    const void* outs[5] = {out_r, out_lse, out_weights, out_r0, out_weights0};
    const int64_t sizes[5] = {r_bytes, lse_bytes, a_bytes, row, (int64_t)T * n * 4};
    const char* names[5] = {"out_r", "out_lse", "out_weights", "out_r0", "out_weights0"};
    for (int i = 3; i < 5; ++i) {
      if (!outs[i]) continue;
      for (int s = 0; s < n; ++s)
        if (overlaps(outs[i], sizes[i], sources[s], row)) return fail(ATTNRES_EINVAL, "%s overlaps source %d", names[i], s);
      for (int j = 0; j < 5; ++j)
        if (j != i && outs[j] && overlaps(outs[i], sizes[i], outs[j], sizes[j]))
          return fail(ATTNRES_EINVAL, "%s overlaps %s", names[i], names[j]);
    }
  }
  if (!twophase_pointers_ok(out_r)) return fail(ATTNRES_EINVAL, "out_r not 16-byte aligned");
  if (out_r0 && !twophase_pointers_ok(out_r0)) return fail(ATTNRES_EINVAL, "out_r0 not 16-byte aligned");
  if (workspace) {
    // the tensor-core logits: the workspace holds the partial dot products;
    // it may not share memory with an input or output
    const int64_t need = interblock_tc_workspace_bytes(n, T, d, dtype, Q);
    if (need < 0) return fail(ATTNRES_ECUDA, "no CUDA device");
    if (need == 0) {
      workspace = nullptr;  // the path does not apply (fp32 sources, d not a multiple of 64): CUDA cores
    } else {
      if (workspace_bytes < need)
        return fail(ATTNRES_EINVAL, "workspace of %lld bytes, %lld needed", (long long)workspace_bytes,
                    (long long)need);
      if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(ATTNRES_EINVAL, "workspace not 256-byte aligned");
      const int64_t row = T * d * (dtype == ATTNRES_BF16 ? 2 : 4);
      for (int s = 0; s < n; ++s)
        if (overlaps(workspace, need, sources[s], row)) return fail(ATTNRES_EINVAL, "workspace overlaps source %d", s);
      if (overlaps(workspace, need, out_r, (int64_t)Q * T * d * 4) ||
          overlaps(workspace, need, out_lse, (int64_t)Q * T * 4) ||
          (out_weights && overlaps(workspace, need, out_weights, (int64_t)Q * T * n * 4)) ||
          (out_r0 && overlaps(workspace, need, out_r0, row)) ||
          (out_weights0 && overlaps(workspace, need, out_weights0, (int64_t)T * n * 4)))
        return fail(ATTNRES_EINVAL, "workspace overlaps an output");
      for (int q = 0; q < Q; ++q)
        if (overlaps(workspace, need, w_queries[q], (int64_t)d * 4))
          return fail(ATTNRES_EINVAL, "workspace overlaps w_queries[%d]", q);
    }
  }
  a.workspace = workspace;
  a.workspace_bytes = workspace ? workspace_bytes : 0;
  a.n = n;
  a.T = T;
  a.d = d;
  a.dtype = dtype;
  a.Q = Q;
  a.eps = eps;
  a.out_r = out_r;
  a.out_lse = out_lse;
  a.out_a = out_weights;
  a.out_r0 = out_r0;
  a.out_a0 = out_weights0;
  a.dev_err = dev_err;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_interblock(a);
  if (e != cudaSuccess) {
    const char* step = interblock_tc_last_step();
    return cuda_fail(e, *step ? step : "attnres_interblock launch");
  }
  return ok();
}

int attnres_intrablock_step(attnres_state* st, const void* F_prev, const float* w_l, int layer_idx,
                            const float* r_inter, const float* lse_inter, const float* a_inter, void* out_r,
                            float* out_weights, int* dev_err, void* stream) {
  int rc = check_state(st);
  if (rc) return rc;
  const int L = st->num_layers, B = st->block_size;
  if (layer_idx < 1 || layer_idx > L) return fail(ATTNRES_EINVAL, "layer_idx %d outside 1..L", layer_idx);
  if (!w_l || !r_inter || !lse_inter || !out_r) return fail(ATTNRES_EINVAL, "w_l/r_inter/lse_inter/out_r is NULL");
  if (!twophase_supported(st->d, st->dtype))
    return fail(ATTNRES_ERANGE, "two-phase schedule needs rows of a 16-byte multiple, at most 2 x 448 vectors");
  const int n = (layer_idx - 1) / B + 1;
  const int i = (layer_idx - 1) % B + 1;
  MergeArgs a{};
  if (i == 1) {
    if (F_prev) return fail(ATTNRES_EINVAL, "first layer of a block: fold the previous block first, F_prev NULL");
    if (st->folded != layer_idx - 1)
      return fail(ATTNRES_ESTATE, "intrablock_step(%d) needs folded == %d, state has %d", layer_idx, layer_idx - 1,
                  st->folded);
  } else {
    if (!F_prev) return fail(ATTNRES_EINVAL, "F_prev is NULL");
    if (st->folded != layer_idx - 2)
      return fail(ATTNRES_ESTATE, "intrablock_step(%d) needs folded == %d, state has %d", layer_idx, layer_idx - 2,
                  st->folded);
    a.prev = i >= 3 ? st->partial : nullptr;
    a.F = F_prev;
    a.dst = st->partial;
  }
  for (const void* q : {a.prev, a.F, (const void*)a.dst, (const void*)r_inter, (const void*)out_r})
    if (!twophase_pointers_ok(q)) return fail(ATTNRES_EINVAL, "two-phase buffers must be 16-byte aligned");
  {
    // r and the weights must not share memory with the state's rows or F
    const int64_t row = st->T * st->d * (st->dtype == ATTNRES_BF16 ? 2 : 4);
    const int64_t a_bytes = st->T * attnres_num_sources(layer_idx, B, L) * 4;
    const void* rows[ATTNRES_MAX_BLOCKS + 3];
    int nr = 0;
    rows[nr++] = st->h0;
    rows[nr++] = st->partial;
    if (F_prev) rows[nr++] = F_prev;
    for (int k = 0; k < num_blocks(L, B); ++k)
      if (st->block_reps[k]) rows[nr++] = st->block_reps[k];
    rc = check_outputs_apart(rows, nr, row, out_r, row, out_weights, a_bytes);
    if (rc != ATTNRES_OK) return rc;
    const int64_t inter_bytes = st->T * st->d * 4;  // the fp32 inter-block aggregate
    if (overlaps(out_r, row, r_inter, inter_bytes) || (out_weights && overlaps(out_weights, a_bytes, r_inter, inter_bytes)))
      return fail(ATTNRES_EINVAL, "an output overlaps r_inter");
  }
  a.w = w_l;
  a.r_inter = r_inter;
  a.lse_inter = lse_inter;
  a.a_inter = a_inter;
  a.out_r = out_r;
  a.out_a = out_weights;
  a.T = st->T;
  a.d = st->d;
  a.dtype = st->dtype;
  a.n = n;
  a.eps = st->eps;
  a.dev_err = dev_err;
  a.stream = static_cast<cudaStream_t>(stream);
  a.early_loads = F_prev && (st->flags & ATTNRES_STATE_EARLY_LOADS) != 0;
  if (st->T > 0) {
    cudaError_t e = launch_merge(a);
    if (e != cudaSuccess) return cuda_fail(e, "attnres_intrablock_step launch");
  }
  if (i >= 2) st->folded = layer_idx - 1;
  return ok();
}

int attnres_state_init(attnres_state* st, const void* h0, void* const* block_reps, int n_block_reps, void* partial,
                       int64_t T, int d, int dtype, int num_layers, int block_size, float eps) {
  if (!st || !h0 || !partial || !block_reps) return fail(ATTNRES_EINVAL, "NULL argument");
  if (!valid_dtype(dtype)) return fail(ATTNRES_EDTYPE, "dtype %d", dtype);
  if (!size_ok(T, d)) return fail(ATTNRES_EINVAL, "T=%lld d=%d", (long long)T, d);
  if (num_layers < 1 || block_size < 1) return fail(ATTNRES_EINVAL, "num_layers/block_size must be >= 1");
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(ATTNRES_EINVAL, "eps must be finite and >= 0");
  const int N = num_blocks(num_layers, block_size);
  if (N > ATTNRES_MAX_BLOCKS) return fail(ATTNRES_ERANGE, "ceil(L/B)=%d > %d", N, ATTNRES_MAX_BLOCKS);
  if (n_block_reps < N) return fail(ATTNRES_EINVAL, "need %d block buffers, got %d", N, n_block_reps);
  // every buffer is one [T, d] row set; none may share memory with another
  // (all checked before the struct is written)
  const int64_t row = T * d * (dtype == ATTNRES_BF16 ? 2 : 4);
  if (overlaps(partial, row, h0, row)) return fail(ATTNRES_EINVAL, "partial overlaps h0");
  for (int k = 0; k < N; ++k) {
    if (!block_reps[k]) return fail(ATTNRES_EINVAL, "block_reps[%d] is NULL", k);
    if (overlaps(block_reps[k], row, partial, row) || overlaps(block_reps[k], row, h0, row))
      return fail(ATTNRES_EINVAL, "block_reps[%d] overlaps h0 or partial", k);
    for (int j = 0; j < k; ++j)
      if (overlaps(block_reps[j], row, block_reps[k], row))
        return fail(ATTNRES_EINVAL, "block_reps[%d] overlaps block_reps[%d]", j, k);
  }
  memset(st, 0, sizeof(*st));
  st->h0 = h0;
  for (int k = 0; k < N; ++k) st->block_reps[k] = block_reps[k];
  st->partial = partial;
  st->T = T;
  st->d = d;
  st->dtype = dtype;
  st->num_layers = num_layers;
  st->block_size = block_size;
  st->eps = eps;
  st->folded = 0;
  st->flags = 0;
  return ok();
}

int attnres_state_resume(attnres_state* st, int folded) {
  int rc = check_state(st);
  if (rc) return rc;
  if (folded < 0 || folded > st->num_layers)
    return fail(ATTNRES_EINVAL, "folded=%d outside 0..L=%d", folded, st->num_layers);
  st->folded = folded;
  return ok();
}

int attnres_state_reset(attnres_state* st) {
  if (!st) return fail(ATTNRES_EINVAL, "state is NULL");
  st->folded = 0;
  return ok();
}

int attnres_num_sources(int layer_idx, int block_size, int num_layers) {
  if (block_size < 1 || num_layers < 1) return fail(ATTNRES_EINVAL, "block_size/num_layers must be >= 1");
  if (layer_idx < 1 || layer_idx > num_layers + 1) return fail(ATTNRES_EINVAL, "layer_idx %d outside 1..L+1", layer_idx);
  if (layer_idx == num_layers + 1) return num_blocks(num_layers, block_size) + 1;
  const int n = (layer_idx - 1) / block_size + 1;
  const int i = (layer_idx - 1) % block_size + 1;
  return n + (i >= 2 ? 1 : 0);
}

int attnres_layer_sources(const attnres_state* st, int layer_idx, const void** out_ptrs, int* out_S) {
  int rc = check_state(st);
  if (rc) return rc;
  if (!out_ptrs || !out_S) return fail(ATTNRES_EINVAL, "NULL output");
  const int L = st->num_layers, B = st->block_size;
  if (layer_idx < 1 || layer_idx > L + 1) return fail(ATTNRES_EINVAL, "layer_idx %d outside 1..L+1", layer_idx);
  if (st->folded != layer_idx - 1)
    return fail(ATTNRES_ESTATE, "layer %d needs %d folded layer outputs, state has %d", layer_idx, layer_idx - 1,
                st->folded);
  *out_S = state_sources(st, out_ptrs);
  return ok();
}

int attnres_block_step(attnres_state* st, const void* F_out, int layer_idx, int* dev_err, void* stream) {
  (void)dev_err;  // the fold kernel has no waits
  int rc = check_state(st);
  if (rc) return rc;
  if (!F_out) return fail(ATTNRES_EINVAL, "F_out is NULL");
  const int L = st->num_layers, B = st->block_size;
  if (layer_idx < 1 || layer_idx > L) return fail(ATTNRES_EINVAL, "layer_idx %d outside 1..L", layer_idx);
  if (st->folded != layer_idx - 1)
    return fail(ATTNRES_ESTATE, "block_step(%d) needs folded == %d, state has %d", layer_idx, layer_idx - 1,
                st->folded);
  {
    // F_out is read while the partial sum or a block sum is written: it may
    // not share memory with any of the state's rows
    const int64_t row = st->T * st->d * (st->dtype == ATTNRES_BF16 ? 2 : 4);
    if (overlaps(F_out, row, st->h0, row) || overlaps(F_out, row, st->partial, row))
      return fail(ATTNRES_EINVAL, "F_out overlaps h0 or partial");
    for (int k = 0; k < num_blocks(L, B); ++k)
      if (st->block_reps[k] && overlaps(F_out, row, st->block_reps[k], row))
        return fail(ATTNRES_EINVAL, "F_out overlaps block_reps[%d]", k);
  }
  const FoldPlan fp = fold_plan(layer_idx, B, L);
  void* dst = fp.ends_block ? st->block_reps[fp.block - 1] : st->partial;
  const void* prev = fp.has_prev ? st->partial : nullptr;
  cudaError_t e = launch_fold(prev, F_out, dst, st->T * (int64_t)st->d, st->dtype, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attnres_block_step launch");
  st->folded = layer_idx;
  return ok();
}

int attnres_layer_step(attnres_state* st, const void* F_prev, const float* w_l, int layer_idx, void* out_r,
                       float* out_weights, int* dev_err, void* stream) {
  int rc = check_state(st);
  if (rc) return rc;
  if (!w_l || !out_r) return fail(ATTNRES_EINVAL, "w_l/out_r is NULL");
  const int L = st->num_layers, B = st->block_size;
  if (layer_idx < 1 || layer_idx > L + 1) return fail(ATTNRES_EINVAL, "layer_idx %d outside 1..L+1", layer_idx);
  if (layer_idx == 1 && F_prev) return fail(ATTNRES_EINVAL, "F_prev must be NULL at layer 1");
  // with F_prev, v_{l-1} is folded here; without, it must have been folded
  // already (layer 1, or a state resumed at a stage boundary)
  const int need = F_prev ? layer_idx - 2 : layer_idx - 1;
  if (st->folded != need)
    return fail(ATTNRES_ESTATE, "layer_step(%d)%s needs folded == %d, state has %d", layer_idx,
                F_prev ? "" : " without F_prev", need, st->folded);
  {
    // r and the weights must not share memory with the state's rows or F
    const int64_t row = st->T * st->d * (st->dtype == ATTNRES_BF16 ? 2 : 4);
    const int64_t a_bytes = st->T * attnres_num_sources(layer_idx, B, L) * 4;
    const void* rows[ATTNRES_MAX_BLOCKS + 3];
    int nr = 0;
    rows[nr++] = st->h0;
    rows[nr++] = st->partial;
    if (F_prev) rows[nr++] = F_prev;
    for (int k = 0; k < num_blocks(L, B); ++k)
      if (st->block_reps[k]) rows[nr++] = st->block_reps[k];
    rc = check_outputs_apart(rows, nr, row, out_r, row, out_weights, a_bytes);
    if (rc != ATTNRES_OK) return rc;
  }

  AggArgs a{};
  a.T = st->T;
  a.d = st->d;
  a.src_dtype = st->dtype;
  a.w = w_l;
  a.eps = st->eps;
  a.out_r = out_r;
  a.out_dtype = st->dtype;
  a.out_a = out_weights;
  a.dev_err = dev_err;
  a.stream = static_cast<cudaStream_t>(stream);
  a.src[0] = st->h0;
  a.n_stored = 1;
  if (!F_prev) {
    a.n_stored = state_sources(st, a.src);
  } else {
    const int p = layer_idx - 1;
    const FoldPlan fp = fold_plan(p, B, L);
    for (int k = 0; k < fp.block - 1; ++k) a.src[a.n_stored++] = st->block_reps[k];
    a.fuse_prev = fp.has_prev ? st->partial : nullptr;
    a.fuse_F = F_prev;
    a.fuse_dst = fp.ends_block ? st->block_reps[fp.block - 1] : st->partial;
    a.early_loads = (st->flags & ATTNRES_STATE_EARLY_LOADS) != 0;
  }
  if (a.S() != attnres_num_sources(layer_idx, B, L))
    return fail(ATTNRES_ESTATE, "internal: source count mismatch at layer %d", layer_idx);
  if (st->T > 0) {
    AggPath path;
    cudaError_t e = launch_aggregate(a, &path);
    if (e != cudaSuccess) return cuda_fail(e, "attnres_layer_step launch");
  }
  st->folded = layer_idx - 1;
  return ok();
}

int attnres_synthetic_layer(const void* x, const float* g, const float* s, void* out, int64_t T, int d, int dtype,
                            void* stream) {
  if (!x || !g || !s || !out) return fail(ATTNRES_EINVAL, "NULL argument");
  if (!valid_dtype(dtype)) return fail(ATTNRES_EDTYPE, "dtype %d", dtype);
  if (!size_ok(T, d)) return fail(ATTNRES_EINVAL, "T=%lld d=%d", (long long)T, d);
  cudaError_t e = launch_synthetic_layer(x, g, s, out, T, d, dtype, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attnres_synthetic_layer launch");
  return ok();
}

int attnres_synthetic_layer_backward(const void* x, const float* g, const float* s, const void* grad_out_a,
                                     const void* grad_out_b, void* grad_x, int64_t T, int d, int dtype, void* stream) {
  if (!valid_dtype(dtype)) return fail(ATTNRES_EDTYPE, "dtype %d", dtype);
  if (!size_ok(T, d)) return fail(ATTNRES_EINVAL, "T=%lld d=%d", (long long)T, d);
  if (T == 0) return ok();
  if (!x || !g || !s || !grad_out_a || !grad_x) return fail(ATTNRES_EINVAL, "NULL argument");
  cudaError_t e = launch_synthetic_layer_backward(x, g, s, grad_out_a, grad_out_b, grad_x, T, d, dtype,
                                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attnres_synthetic_layer_backward launch");
  return ok();
}

int attnres_debug_wait_test(uint64_t wait_limit_ns, int withhold_row) {
  if (withhold_row < -1 || withhold_row > 7) return fail(ATTNRES_EINVAL, "withhold_row %d", withhold_row);
  set_debug_wait_test((unsigned long long)wait_limit_ns, withhold_row);
  return ok();
}

int attnres_fold(const void* prev, const void* F, void* dst, int64_t T, int d, int dtype, void* stream) {
  if (!valid_dtype(dtype)) return fail(ATTNRES_EDTYPE, "dtype %d", dtype);
  if (!size_ok(T, d)) return fail(ATTNRES_EINVAL, "T=%lld d=%d", (long long)T, d);
  if (T == 0) return ok();
  if (!F || !dst) return fail(ATTNRES_EINVAL, "NULL argument");
  cudaError_t e = launch_fold(prev, F, dst, T * (int64_t)d, dtype, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attnres_fold launch");
  return ok();
}

}  // extern "C"
