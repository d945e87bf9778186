// Depth-wise attention over the sources of one layer (Block AttnRes).
//
// Per token t, with S sources h_s = src_s[t, :] of d channels and the
// layer's pseudo-query w ("Kimi K3 deep-dive series (2): AttnRes and Stable
// LatentMoE", §2; eps from "Kimi K3 model structure (6)", odd facts):
//     z_s = (w . h_s) / sqrt(mean_c h_s[c]^2 + eps)     (w . RMSNorm(h_s))
//     a   = softmax_s(z)
//     r   = sum_s a_s h_s                                (raw sources)
// All arithmetic is fp32; bf16 is a storage format only.
//
// Kernels:
//
//  agg_ring_kernel  (the hot path: S <= 9, 16-byte aligned rows of at most
//      2 x 448 16-byte vectors, e.g. d = 7168 bf16).  One persistent CTA per
//      SM.  A producer warp streams every source row of the CTA's tokens
//      into a ring of shared-memory slots with TMA bulk copies
//      (cp.async.bulk, completion on an mbarrier per slot).  448 consumer
//      threads each own the same 16-byte vectors of every row: they copy
//      their vectors of each landed row into registers and release the slot
//      at once, so the ring (up to ~225 KB per SM) is almost entirely bytes
//      in flight.  Dot products and sums of squares for all S sources are
//      reduced with a warp reduce-scatter and one cross-warp step (one named
//      barrier per token); the weighted sum is then formed from registers.
//      Every source byte is read from HBM exactly once.  The kernel template
//      is in ring_kernel.cuh (bf16 rows of d = 7168 get one instantiation
//      per source count, ring_fixed_s.cu / ring_fixed_s_fused.cu); the
//      shared layout, vector packing and producer live in ring_common.cuh.
//      This file holds the dispatch and the generic kernel.
//
//  agg_ring_multi_kernel (aggregate_multi.cu: 10 <= S <= 128, same rows):
//      the same ring, sources taken in groups of 6 or 9 with an online
//      softmax.
//
//  agg_split_kernel (aggregate_split.cu, opt-in with ATTNRES_SPLIT=1): few
//      tokens, each shared by a thread-block cluster of 2-8 CTAs.
//
//  agg_generic_kernel  (everything else: any d, any pointer alignment, fp32
//      rows too wide for registers).  One CTA per token, plain loads, two
//      passes over the token's rows (the second mostly from L2).
//
// Both can fuse the block bookkeeping: the last source is formed on the fly
// as round(prev + F) (or F), written out as the new partial sum / block
// representation, and used, already rounded, as a source.
#include <math.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>

#include "attnres.h"
#include "device_common.cuh"
#include "launch.h"
#include "ring_common.cuh"
#include "ring_kernel.cuh"

namespace attnres {

// --------------------------------------------------------- generic kernel --

constexpr int kGenThreads = 256;

struct GenericParams {
  const char* src[kMaxSources];
  const char* fuse_prev;
  const char* fuse_F;
  char* fuse_dst;
  const float* w;
  char* out_r;
  float* out_a;
  long long T;
  int d;
  int n_stored;
  int S;
  float eps;
};

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kGenThreads) agg_generic_kernel(const __grid_constant__ GenericParams p) {
  __shared__ float s_red[kGenThreads / 32][2];
  __shared__ float s_za[kMaxSources];  // logits, then weights
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d = p.d, S = p.S;
  pdl_wait();
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done
  for (long long t = blockIdx.x; t < p.T; t += gridDim.x) {
    const long long row = t * (long long)d;
    // pass 1: logit of every source (forming the fused source on the way)
    for (int s = 0; s < S; ++s) {
      float dot = 0.f, ss = 0.f;
      if (s < p.n_stored) {
        const Tin* h = reinterpret_cast<const Tin*>(p.src[s]) + row;
        for (int c = tid; c < d; c += kGenThreads) {
          const float x = load_elem(h + c);
          dot = fmaf(p.w[c], x, dot);
          ss = fmaf(x, x, ss);
        }
      } else {
        const Tin* F = reinterpret_cast<const Tin*>(p.fuse_F) + row;
        const Tin* P = p.fuse_prev ? reinterpret_cast<const Tin*>(p.fuse_prev) + row : nullptr;
        Tin* D = reinterpret_cast<Tin*>(p.fuse_dst) + row;
        for (int c = tid; c < d; c += kGenThreads) {
          float x = load_elem(F + c);
          if (P) x = round_to<Tin>(load_elem(P + c) + x);
          store_elem(D + c, x);
          dot = fmaf(p.w[c], x, dot);
          ss = fmaf(x, x, ss);
        }
      }
      dot = warp_sum(dot);
      ss = warp_sum(ss);
      if (lane == 0) {
        s_red[warp][0] = dot;
        s_red[warp][1] = ss;
      }
      __syncthreads();
      if (tid == 0) {
        float dd = 0.f, sq = 0.f;
#pragma unroll
        for (int w = 0; w < kGenThreads / 32; ++w) {
          dd += s_red[w][0];
          sq += s_red[w][1];
        }
        s_za[s] = dd / sqrtf(sq / (float)d + p.eps);
      }
      __syncthreads();
    }
    // depth softmax over the S logits
    if (warp == 0) {
      float m = -INFINITY;
      for (int s = lane; s < S; s += 32) m = fmaxf(m, s_za[s]);
      m = warp_max(m);
      float tot = 0.f;
      for (int s = lane; s < S; s += 32) tot += expf(s_za[s] - m);
      tot = warp_sum(tot);
      for (int s = lane; s < S; s += 32) {
        const float a = expf(s_za[s] - m) / tot;
        s_za[s] = a;
        if (p.out_a) p.out_a[t * S + s] = a;
      }
    }
    __syncthreads();
    // pass 2: weighted sum of the raw sources
    for (int c = tid; c < d; c += kGenThreads) {
      float acc = 0.f;
      for (int s = 0; s < S; ++s) {
        const Tin* h = (s < p.n_stored) ? reinterpret_cast<const Tin*>(p.src[s]) + row
                                        : reinterpret_cast<const Tin*>(p.fuse_dst) + row;
        acc = fmaf(s_za[s], load_elem(h + c), acc);
      }
      store_elem(reinterpret_cast<Tout*>(p.out_r) + row + c, acc);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- launch --

cudaError_t device_info(DeviceInfo* info) {
  constexpr int kMaxDevices = 64;
  static DeviceInfo cache[kMaxDevices];
  static std::atomic<bool> have[kMaxDevices];  // set after cache[dev] is filled
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices && have[dev]) {
    *info = cache[dev];
    return cudaSuccess;
  }
  DeviceInfo di{};
  e = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&di.l2_bytes, cudaDevAttrL2CacheSize, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices) {
    cache[dev] = di;
    have[dev] = true;
  }
  *info = di;
  return cudaSuccess;
}

unsigned long long current_context_id() {
  using GetCurrent = int (*)(void**);
  using GetId = int (*)(void*, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  if (!get_current || !get_id) return 0;
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != 0 || !ctx) return 0;
  if (get_id(ctx, &id) != 0) return 0;
  return id;
}

cudaError_t SmemOptIn::ensure(const void* kern, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool slot = dev >= 0 && dev < kMaxDevices;
  const unsigned long long now = current_context_id();
  if (slot && now != 0 && ctx[dev].load() == now) return cudaSuccess;
  DeviceInfo di;
  e = device_info(&di);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes > 0 ? bytes : di.max_smem_optin);
  if (e != cudaSuccess) return e;
  if (slot) ctx[dev].store(current_context_id());  // the call above made the context current
  return cudaSuccess;
}

template <typename Tin, typename Tout>
static cudaError_t launch_ring_vpt(const RingParams& rp, int vpt, bool fused, int grid, int smem,
                                   cudaStream_t stream) {
  const bool exact = rp.nvec == vpt * kRingConsumers;
  if constexpr (sizeof(Tin) == 2 && sizeof(Tout) == 2) {
    // bf16 storage at d = 7168 (the K3 width): one kernel per source count
    if (exact && vpt == 2 && rp.S >= 1 && rp.S <= kRingSmax)
      return !fused ? launch_ring_fixed_s(rp, grid, smem, stream)
             : rp.fuse_prev ? launch_ring_fixed_s_fused_prev(rp, grid, smem, stream)
                            : launch_ring_fixed_s_fused_noprev(rp, grid, smem, stream);
  }
  if (vpt == 1) {
    return fused ? launch_ring_t<Tin, Tout, 1, true, false>(rp, grid, smem, stream)
                 : launch_ring_t<Tin, Tout, 1, false, false>(rp, grid, smem, stream);
  }
  if (exact) {
    return fused ? launch_ring_t<Tin, Tout, 2, true, true>(rp, grid, smem, stream)
                 : launch_ring_t<Tin, Tout, 2, false, true>(rp, grid, smem, stream);
  }
  return fused ? launch_ring_t<Tin, Tout, 2, true, false>(rp, grid, smem, stream)
               : launch_ring_t<Tin, Tout, 2, false, false>(rp, grid, smem, stream);
}

template <typename Tin, typename Tout>
static cudaError_t launch_generic_t(const GenericParams& gp, int grid, cudaStream_t stream) {
  const cudaError_t e = launch_kernel(agg_generic_kernel<Tin, Tout>, dim3(grid), dim3(kGenThreads), 0, stream, gp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

static std::atomic<unsigned long long> g_wait_limit_ns{0};
static std::atomic<int> g_withhold_row1{0};

void set_debug_wait_test(unsigned long long ns, int withhold_row) {
  g_wait_limit_ns.store(ns);
  g_withhold_row1.store(withhold_row + 1);
}

int debug_withhold_row1() { return g_withhold_row1.load(); }

unsigned long long wait_limit_ns() {
  const unsigned long long v = g_wait_limit_ns.load();
  return v ? v : kWaitLimitNs;
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("ATTNRES_NO_PDL");
    return !(v && v[0] && v[0] != '0');
  }();
  return on;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaError_t launch_aggregate(const AggArgs& a, AggPath* path) {
  *path = kPathNone;
  if (a.T <= 0) return cudaSuccess;
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;

  const bool in_bf16 = a.src_dtype == ATTNRES_BF16;
  const bool out_bf16 = a.out_dtype == ATTNRES_BF16;
  const int esz = in_bf16 ? 2 : 4;
  const int osz = out_bf16 ? 2 : 4;
  const int S = a.S();
  const bool fused = a.fuse_F != nullptr;
  const long long row_bytes = (long long)a.d * esz;
  const int epv = 16 / esz;

  // ---- can a ring kernel take it?  (S <= 9: one group per token; up to
  // 128: groups of 9 with an online softmax; few tokens: a cluster per token)
  bool aligned = S <= kMaxSources && row_bytes % 16 == 0;
  const long long nvec = row_bytes / 16;
  for (int s = 0; aligned && s < a.n_stored; ++s) aligned = aligned16(a.src[s]);
  if (aligned && fused)
    aligned = aligned16(a.fuse_F) && aligned16(a.fuse_dst) && (!a.fuse_prev || aligned16(a.fuse_prev));
  const int out_store = epv * osz > 16 ? 16 : epv * osz;  // widest single store of an output vector
  if (aligned) aligned = (reinterpret_cast<uintptr_t>(a.out_r) % out_store) == 0;
  const int split_c = aligned && S <= kRingSmax ? split_cluster_size(a.T, di.sm_count, nvec) : 0;
  const int vpt = (int)((nvec + kRingConsumers - 1) / kRingConsumers);
  bool ring = aligned && vpt >= 1 && vpt <= kRingMaxVpt;
  int nslots = 0;
  if (ring) {
    const long long avail = (long long)di.max_smem_optin - kRingHeaderBytes;
    nslots = (int)(avail / row_bytes);
    if (nslots > kRingMaxSlots) nslots = kRingMaxSlots;
    ring = nslots >= 1;
  }

  if (ring || split_c > 0) {
    RingParams rp{};
    for (int s = 0; s < a.n_stored; ++s) rp.src[s] = static_cast<const char*>(a.src[s]);
    rp.fuse_prev = static_cast<const char*>(a.fuse_prev);
    rp.fuse_F = static_cast<const char*>(a.fuse_F);
    rp.fuse_dst = static_cast<char*>(a.fuse_dst);
    rp.w = a.w;
    rp.out_r = static_cast<char*>(a.out_r);
    rp.out_a = a.out_a;
    rp.dev_err = a.dev_err;
    rp.T = a.T;
    rp.d = a.d;
    rp.n_stored = a.n_stored;
    rp.S = S;
    rp.nvec = (int)nvec;
    rp.row_bytes = (int)row_bytes;
    rp.out_row_bytes = (int)((long long)a.d * osz);
    rp.nslots = nslots;
    rp.eps = a.eps;
    rp.inv_d = 1.0f / (float)a.d;
    rp.wait_ns = wait_limit_ns();
    rp.withhold_row1 = debug_withhold_row1();
    // a fused step keeps source 0 (h_0, read by every layer) in L2 only
    // while all of its rows fit in half of L2; beyond that the marked lines
    // would crowd out the rest, and every row takes the default policy
    rp.keep_src0 = fused && a.T * (long long)row_bytes <= (long long)di.l2_bytes / 2;
    rp.early_loads = fused && a.early_loads ? 1 : 0;
    if (split_c > 0) {
      *path = kPathRingSplit;
      return launch_ring_split(rp, split_c, fused, in_bf16, out_bf16, di.sm_count, di.max_smem_optin, a.stream);
    }
    const int grid = (int)(a.T < di.sm_count ? a.T : di.sm_count);
    const int smem = kRingHeaderBytes + nslots * (int)row_bytes;
    if (S > kRingSmax) {
      *path = kPathRingMulti;
      return launch_ring_multi(rp, vpt, fused, rp.nvec == vpt * kRingConsumers, in_bf16, out_bf16, grid, smem,
                               a.stream);
    }
    *path = kPathRing;
    if (in_bf16) {
      return out_bf16 ? launch_ring_vpt<bf16_t, bf16_t>(rp, vpt, fused, grid, smem, a.stream)
                      : launch_ring_vpt<bf16_t, float>(rp, vpt, fused, grid, smem, a.stream);
    }
    return out_bf16 ? launch_ring_vpt<float, bf16_t>(rp, vpt, fused, grid, smem, a.stream)
                    : launch_ring_vpt<float, float>(rp, vpt, fused, grid, smem, a.stream);
  }

  GenericParams gp{};
  for (int s = 0; s < a.n_stored; ++s) gp.src[s] = static_cast<const char*>(a.src[s]);
  gp.fuse_prev = static_cast<const char*>(a.fuse_prev);
  gp.fuse_F = static_cast<const char*>(a.fuse_F);
  gp.fuse_dst = static_cast<char*>(a.fuse_dst);
  gp.w = a.w;
  gp.out_r = static_cast<char*>(a.out_r);
  gp.out_a = a.out_a;
  gp.T = a.T;
  gp.d = a.d;
  gp.n_stored = a.n_stored;
  gp.S = S;
  gp.eps = a.eps;
  const long long max_grid = (long long)di.sm_count * 8;
  const int grid = (int)(a.T < max_grid ? a.T : max_grid);
  *path = kPathGeneric;
  if (in_bf16) {
    return out_bf16 ? launch_generic_t<bf16_t, bf16_t>(gp, grid, a.stream)
                    : launch_generic_t<bf16_t, float>(gp, grid, a.stream);
  }
  return out_bf16 ? launch_generic_t<float, bf16_t>(gp, grid, a.stream)
                  : launch_generic_t<float, float>(gp, grid, a.stream);
}

}  // namespace attnres
