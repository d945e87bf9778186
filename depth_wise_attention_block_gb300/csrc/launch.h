// Host-side launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <atomic>

#include <cuda_runtime.h>
#include <stdint.h>

namespace attnres {

constexpr int kMaxSources = 128;

// One aggregation launch, possibly with the block bookkeeping fused in.
//
// Stored sources src[0 .. n_stored-1] are read as they are.  When fuse_F is
// non-null one more source follows them, formed on the fly as
//     x = round(fuse_prev + fuse_F)   (or fuse_F alone when fuse_prev is null)
// written to fuse_dst and used, already rounded, as source n_stored.
struct AggArgs {
  const void* src[kMaxSources];
  int n_stored;
  const void* fuse_prev;
  const void* fuse_F;
  void* fuse_dst;
  int64_t T;
  int d;
  int src_dtype;  // attnres_dtype (stored sources, fused rows, fuse_dst)
  const float* w;
  float eps;
  void* out_r;
  int out_dtype;
  float* out_a;   // [T, S] or null
  int* dev_err;
  cudaStream_t stream;
  bool early_loads;  // fused: stored rows of the first token loaded before the previous kernel ends

  int S() const { return n_stored + (fuse_F ? 1 : 0); }
};

// Which kernel a launch took (for tests and the bench).
enum AggPath { kPathNone = 0, kPathRing = 1, kPathGeneric = 2, kPathRingMulti = 3, kPathRingSplit = 4 };

// Launch; returns cudaSuccess or the launch error.  *path gets the kernel.
cudaError_t launch_aggregate(const AggArgs& a, AggPath* path);

// Two-phase schedule (twophase.cu).
constexpr int kMaxQueries = 16;
struct InterArgs {
  const void* src[kMaxSources];
  int n;  // cached sources, <= 9
  int64_t T;
  int d;
  int dtype;
  const float* wq[kMaxQueries];
  int Q;
  float eps;
  float* out_r;    // [Q, T, d]
  float* out_lse;  // [Q, T]
  float* out_a;    // [Q, T, n] or null
  void* out_r0;    // [T, d] of dtype or null: query 0's row rounded, a block's first layer
  float* out_a0;   // [T, n] or null: query 0's weights
  void* workspace;  // the tensor-core logits' scratch (interblock_tc_workspace_bytes), or null
  int64_t workspace_bytes;
  int* dev_err;
  cudaStream_t stream;
};
// the queries of one inter-block pass, as a kernel parameter
struct InterQueries {
  const float* w[kMaxQueries];
};
struct MergeArgs {
  const void* prev;
  const void* F;
  void* dst;
  const float* w;
  const float* r_inter;
  const float* lse_inter;
  const float* a_inter;
  void* out_r;
  float* out_a;
  int64_t T;
  int d;
  int dtype;
  int n;
  float eps;
  int* dev_err;  // the ring merge's bounded waits (bf16 rows of 2 x 448 vectors)
  cudaStream_t stream;
  bool early_loads;  // the ring merge: prev and r_inter of the first token loaded before the previous kernel ends
};
bool twophase_supported(int d, int dtype);
bool twophase_pointers_ok(const void* p);
cudaError_t launch_interblock(const InterArgs& a);
// The inter-block logits on the tensor cores (twophase_tc.cu): bf16 sources
// with d a multiple of 64.  Workspace bytes for n sources, T tokens and Q
// queries on the current device (0: the path does not apply; -1: error).
bool interblock_tc_supported(int n, int d, int dtype);
int64_t interblock_tc_workspace_bytes(int n, long long T, int d, int dtype, int Q);
// Splits the queries into bf16 terms and computes the partial dot products
// [ksplit][T][n][Q] into the workspace; returns where they are.
cudaError_t launch_interblock_tc(const InterArgs& a, void* workspace, float** dots, int* ksplit);
// the step of the last launch_interblock_tc that failed on this thread ("" if none)
const char* interblock_tc_last_step();
cudaError_t launch_merge(const MergeArgs& a);

// Backward of one aggregation (see backward.cu).
struct BwdArgs {
  const void* src[kMaxSources];
  void* grad_src[kMaxSources];
  int S;
  int64_t T;
  int d;
  int dtype;  // of sources, grad_r and grad_src
  const float* w;
  float eps;
  const void* grad_r;
  bool accumulate;
  float* grad_w;
  float* workspace;  // [backward_blocks(T), d] fp32
  int* dev_err;
  cudaStream_t stream;
};
cudaError_t launch_aggregate_backward(const BwdArgs& a);
// CTAs (= fp32 workspace rows of d floats) the backward uses for T tokens
int64_t backward_blocks(int64_t T);
// Device address and size (floats) of the library's own backward scratch
// array on the current device (backward.cu).
cudaError_t noalloc_backward_scratch(float** ptr, int64_t* capacity_floats);

// dst = prev ? round(prev + F) : F over n = T*d elements of dtype.
cudaError_t launch_fold(const void* prev, const void* F, void* dst, int64_t n, int dtype,
                        cudaStream_t stream);

// out = round(tanh(x * g[c]) * s[c]) over [T, d].
cudaError_t launch_synthetic_layer(const void* x, const float* g, const float* s, void* out,
                                   int64_t T, int d, int dtype, cudaStream_t stream);
cudaError_t launch_synthetic_layer_backward(const void* x, const float* g, const float* s, const void* dva,
                                            const void* dvb, void* dx, int64_t T, int d, int dtype,
                                            cudaStream_t stream);

// Launch `kern` with programmatic stream serialization allowed (the kernel
// may start while the previous kernel on the stream finishes; every kernel
// here waits for it with griddepcontrol.wait before touching global memory).
// Set ATTNRES_NO_PDL=1 in the environment to launch plainly.
bool pdl_enabled();

// The bounded-wait test (attnres_debug_wait_test): the limit of each
// main-loop wait in the ring kernels (2 s by default; the final drain always
// keeps 2 s) and 1 + the row each CTA's producer arms without a copy (0 =
// none).
unsigned long long wait_limit_ns();
int debug_withhold_row1();
void set_debug_wait_test(unsigned long long ns, int withhold_row);

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Per-device properties, cached.
struct DeviceInfo {
  int sm_count;
  int max_smem_optin;
  int l2_bytes;
};
cudaError_t device_info(DeviceInfo* info);

// Unique id of the calling thread's current CUDA context, 0 if none is
// current yet or the driver lacks the entry points (cuCtxGetCurrent and
// cuCtxGetId, reached through cudaGetDriverEntryPointByVersion).  A context
// torn down and created again (cudaDeviceReset) gets a new id.
unsigned long long current_context_id();

// The large dynamic shared-memory opt-in of one kernel
// (cudaFuncAttributeMaxDynamicSharedMemorySize), set once per device and
// context: a context recreated after cudaDeviceReset reloads the module
// without it, so a new context id sets it again.
struct SmemOptIn {
  static constexpr int kMaxDevices = 64;
  std::atomic<unsigned long long> ctx[kMaxDevices];  // context the attribute was set in (0: not yet)
  // bytes: the dynamic shared memory the kernel's launches use, or 0 for the
  // device's whole opt-in size (kernels without static shared memory)
  cudaError_t ensure(const void* kern, int bytes = 0);
};

}  // namespace attnres
