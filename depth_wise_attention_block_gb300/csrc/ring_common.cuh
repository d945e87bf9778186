// Pieces shared by the ring kernels of libattnres (ring_kernel.cuh: one
// group of at most 9 sources per token; aggregate_multi.cu: any number of
// sources in groups with an online softmax; aggregate_split.cu and
// twophase.cu: variants): the shared-memory layout, the kernel parameters,
// 16-byte vector packing, the warp reduce-scatter of the per-source partial
// sums, output stores, the TMA producer and its drain.
#pragma once

#include "attnres.h"
#include "device_common.cuh"
#include "launch.h"

namespace attnres {

// ------------------------------------------------------------ ring kernel --

constexpr int kRingConsumerWarps = 14;
constexpr int kRingConsumers = kRingConsumerWarps * 32;  // 448
constexpr int kRingThreads = kRingConsumers + 32;        // + one producer warp
constexpr int kRingSmax = 9;                             // K3: embedding + 7 blocks + partial
constexpr int kRingMaxVpt = 2;                           // 16-byte vectors per thread per row
constexpr int kRingMaxSlots = 16;
constexpr int kRingBarrierId = 1;                        // named barrier of the consumers

struct RingShared {
  uint64_t full[kRingMaxSlots];   // slot holds a landed row
  uint64_t empty[kRingMaxSlots];  // every consumer warp has taken its part of the row
  // per-warp totals of dot(w, h_s) and sum(h_s^2), double-buffered by the
  // token loop's iteration parity (one barrier per token suffices)
  float red[2][kRingConsumerWarps][2 * kRingSmax];
  // set (never cleared) when a wait of the token loop's iteration i gave up;
  // indexed by i & 1 so a fast warp flagging iteration i+1 cannot be seen
  // by a slow warp still reading the flag of iteration i
  int abort_flag[2];
  uint64_t wait_ns;  // copy of RingParams::wait_ns (read by the consumers' slow waits)
  float zbuf[kMaxSources];  // logits of the token in flight (multi-group kernel)
};
constexpr int kRingHeaderBytes = (int)((sizeof(RingShared) + 127) / 128 * 128);

struct RingParams {
  unsigned long long wait_ns;  // limit of each main-loop wait (the final drain keeps the default)
  int pad_rows;                // rows appended to each token (re-reads of src[0]'s row; multi-group kernel)
  int withhold_row1;           // bounded-wait test: 1 + the row of each CTA's first token armed
                               // without a copy (its waits must run out); 0 = none
  int keep_src0;               // fused step whose source 0 fits in L2: keep it there, stream the rest
  int early_loads;             // fused step: the first token's stored rows are loaded before the wait
                               // for the previous kernel (only F needs that kernel)
  const char* src[kMaxSources];
  const char* fuse_prev;
  const char* fuse_F;
  char* fuse_dst;
  const float* w;
  char* out_r;
  float* out_a;
  int* dev_err;
  long long T;
  int d;
  int n_stored;
  int S;
  int nvec;       // 16-byte vectors per source row
  int row_bytes;  // bytes per source row
  int out_row_bytes;
  int nslots;
  float eps;
  float inv_d;    // 1/d rounded to fp32
};

template <typename Tin>
struct Vec;
template <>
struct Vec<bf16_t> {
  static constexpr int kElems = 8;
  static __device__ __forceinline__ void unpack(const uint4& v, float* f) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
    f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
    f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
  }
  static __device__ __forceinline__ uint4 pack(const float* f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
  }
  // the 8 values as 4 packed fp32 pairs
  static __device__ __forceinline__ void pairs(const uint4& v, uint64_t* p) {
    p[0] = f2_pack(bf16lo(v.x), bf16hi(v.x));
    p[1] = f2_pack(bf16lo(v.y), bf16hi(v.y));
    p[2] = f2_pack(bf16lo(v.z), bf16hi(v.z));
    p[3] = f2_pack(bf16lo(v.w), bf16hi(v.w));
  }
};
template <>
struct Vec<float> {
  static constexpr int kElems = 4;
  static __device__ __forceinline__ void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
  static __device__ __forceinline__ void pairs(const uint4& v, uint64_t* p) {
    p[0] = f2_pack(__uint_as_float(v.x), __uint_as_float(v.y));
    p[1] = f2_pack(__uint_as_float(v.z), __uint_as_float(v.w));
  }
};

// One level of a reduce-scatter over the warp: N values per lane; lanes
// whose bit OFF is clear keep values [0, K), the others [K, N) (padded to
// M values); each exchanges what it does not keep with lane ^ OFF.
template <int N, int K, int OFF>
__device__ __forceinline__ void rs_level(float* v, int lane) {
  constexpr int M = K > N - K ? K : N - K;
  const bool up = (lane & OFF) != 0;
  float out[M];
#pragma unroll
  for (int i = 0; i < M; ++i) {
    const float lo_part = i < K ? v[i] : 0.f;
    const float hi_part = K + i < N ? v[K + i] : 0.f;
    const float keep = up ? hi_part : lo_part;
    const float send = up ? lo_part : hi_part;
    out[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
  }
#pragma unroll
  for (int i = 0; i < M; ++i) v[i] = out[i];
}

// 18 partials (dot and sum of squares of 9 sources) summed over the warp in
// 20 shuffles (18 -> 9 -> 5 -> 3 -> 2 -> 1 values per lane).  Afterwards the
// lanes of kRsValidLanes hold, in v[0], the warp total of value rs_index(lane).
constexpr uint32_t kRsValidLanes = 0x17371737u;
__device__ __forceinline__ int rs_index(int lane) {
  return 9 * ((lane >> 4) & 1) + 5 * ((lane >> 3) & 1) + 3 * ((lane >> 2) & 1) + 2 * ((lane >> 1) & 1) +
         (lane & 1);
}
__device__ __forceinline__ void reduce_scatter18(float* v, int lane) {
  rs_level<18, 9, 16>(v, lane);
  rs_level<9, 5, 8>(v, lane);
  rs_level<5, 3, 4>(v, lane);
  rs_level<3, 2, 2>(v, lane);
  rs_level<2, 1, 1>(v, lane);
}


// Generic reduce-scatter of N <= 32 per-lane values over the warp, halving
// the kept range at each of the offsets 16, 8, 4, 2, 1 (lower lanes keep the
// first ceil(n/2) values).  Afterwards lane `lane` holds in v[0] the warp
// total of value rs_lane_index<N>(lane), if rs_lane_valid<N>(lane).
template <int N, int OFF>
__device__ __forceinline__ void rs_levels(float* v, int lane) {
  if constexpr (OFF >= 1) {
    if constexpr (N > 1) {
      constexpr int K = (N + 1) / 2;
      rs_level<N, K, OFF>(v, lane);
      rs_levels<K, OFF / 2>(v, lane);
    } else {
      // one value left per lane: the remaining levels sum it pairwise
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
      rs_levels<1, OFF / 2>(v, lane);
    }
  }
}
template <int N>
__device__ __forceinline__ void reduce_scatter(float* v, int lane) {
  rs_levels<N, 16>(v, lane);
}
// The same after its first level (offset 16, lower lanes keeping values
// [0, (N+1)/2)) was done by the caller: v holds (N+1)/2 values per lane.
template <int N>
__device__ __forceinline__ void reduce_scatter_after_first(float* v, int lane) {
  rs_levels<(N + 1) / 2, 8>(v, lane);
}
// Size of the kept half at level `level` (0: offset 16 ... 4: offset 1) of
// reduce_scatter<N>; it does not depend on which half a lane keeps.
__host__ __device__ constexpr int rs_split(int N, int level) {
  int n = N, K = 0;
  for (int i = 0; i <= level; ++i) {
    K = (n + 1) / 2;
    n = K;
  }
  return K;
}
// Lanes left holding a value after reduce_scatter<N> (the others hold
// padding or a duplicate).
__host__ __device__ constexpr uint32_t rs_valid_mask(int N) {
  uint32_t m = 0;
  for (int lane = 0; lane < 32; ++lane) {
    int n = N, len = N;
    for (int off = 16; off >= 1; off >>= 1) {
      const int K = (n + 1) / 2;
      if (lane & off) len = len > K ? len - K : 0;
      else len = len < K ? len : K;
      n = K;
    }
    if (len >= 1) m |= 1u << lane;
  }
  return m;
}
template <int N>
struct RsMap {
  static constexpr uint32_t kValid = rs_valid_mask(N);
  static constexpr int K0 = rs_split(N, 0), K1 = rs_split(N, 1), K2 = rs_split(N, 2), K3 = rs_split(N, 3),
                       K4 = rs_split(N, 4);
};
// index held by a lane after reduce_scatter<N>, or -1 if it holds padding:
// the upper half taken at a level adds that level's kept size
template <int N>
__device__ __forceinline__ int rs_lane_index(int lane) {
  using M = RsMap<N>;
  const int idx = M::K0 * ((lane >> 4) & 1) + M::K1 * ((lane >> 3) & 1) + M::K2 * ((lane >> 2) & 1) +
                  M::K3 * ((lane >> 1) & 1) + M::K4 * (lane & 1);
  return ((M::kValid >> lane) & 1u) ? idx : -1;
}
static_assert(RsMap<18>::kValid == kRsValidLanes, "the 18-value map of the general form");

// store EPV output values of vector `vec` of an output row
template <typename Tout, int EPV>
__device__ __forceinline__ void store_out(char* row, int vec, const float* acc) {
  if constexpr (sizeof(Tout) == 2 && EPV == 8) {
    *reinterpret_cast<uint4*>(row + (size_t)vec * 16) = Vec<bf16_t>::pack(acc);
  } else if constexpr (sizeof(Tout) == 2 && EPV == 4) {
    *reinterpret_cast<uint2*>(row + (size_t)vec * 8) =
        make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
  } else if constexpr (sizeof(Tout) == 4 && EPV == 8) {
    uint4* o = reinterpret_cast<uint4*>(row + (size_t)vec * 32);
    o[0] = Vec<float>::pack(acc);
    o[1] = Vec<float>::pack(acc + 4);
  } else {
    *reinterpret_cast<uint4*>(row + (size_t)vec * 16) = Vec<float>::pack(acc);
  }
}


// Every issued copy must have landed before a CTA exits: wait on the latest
// armed phase of each slot (already-consumed phases pass at once).  The
// one row the bounded-wait test arms without a copy is skipped: its slot is
// never released (its waits run out), so that phase is still its latest.
__device__ __forceinline__ void ring_drain(uint64_t* full, int nslots, long long issued, int withhold_row1) {
  const long long armed_slots = issued < nslots ? issued : nslots;
  for (int k = 0; k < armed_slots; ++k) {
    const long long uses = (issued - 1 - k) / nslots + 1;
    if (uses == 1 && k + 1 == withhold_row1) continue;
    mbar_wait_bounded(smem_addr(&full[k]), (uint32_t)((uses - 1) & 1));
  }
}

// The producer: one thread streams every source row of this CTA's tokens
// (t = blockIdx.x, blockIdx.x + gridDim.x, ...) into the ring, in order,
// each row one TMA bulk copy completing on its slot's `full` barrier, after
// the slot's previous row was released by all consumer warps.  On a wait
// that runs out it stops issuing; in every case it waits (bounded) for its
// copies in flight before returning, so the CTA never exits under a copy.
// It waits for the previous kernel (pdl_wait) before its first row, or,
// with early_loads, only before the first token's F row: the stored rows
// (h_0, the block sums, the previous partial sum) were written two or more
// launches back, which have completed when this kernel starts.
__device__ __forceinline__ void ring_produce(const RingParams& p, RingShared& sh, uint32_t ring) {
  const int nslots = p.nslots;
  const long long T = p.T;
  const bool fused = p.fuse_F != nullptr;
  const int real_rows = p.n_stored + (fused ? (p.fuse_prev ? 2 : 1) : 0);
  const int rows = real_rows + p.pad_rows;
  uint32_t slot = 0, lap = 0;
  long long issued = 0;
  bool ok = true;
  // A fused layer step runs inside a stack, where source 0 (the embedding
  // h_0) is read again by every layer: while h_0 fits in half of L2
  // (keep_src0) its rows are kept there and every other row streams
  // through once (evict first), which also spares the rows the previous
  // kernels just wrote.  A single aggregation, or a fused step over more
  // tokens, streams everything with the default policy.
  const uint64_t keep = l2_policy_evict_last(), stream = l2_policy_evict_first();
  bool waited = false;
  for (long long t = blockIdx.x; t < T && ok; t += gridDim.x) {
    const long long off = t * (long long)p.row_bytes;
    for (int j = 0; j < rows; ++j) {
      if (!waited && !(p.early_loads && t == blockIdx.x && j != real_rows - 1)) {
        pdl_wait();
        pdl_trigger();
        waited = true;
      }
      const char* g;
      if (j < p.n_stored) g = p.src[j] + off;
      else if (j >= real_rows) g = p.src[0] + off;  // padding: source 0's row again
      else if (p.fuse_prev && j == p.n_stored) g = p.fuse_prev + off;
      else g = p.fuse_F + off;
      // first lap: parity 1 of a fresh barrier counts as complete
      if (!mbar_wait_bounded(smem_addr(&sh.empty[slot]), (lap & 1u) ^ 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      const uint32_t full = smem_addr(&sh.full[slot]);
      mbar_arrive_expect_tx(full, (uint32_t)p.row_bytes);
      // the bounded-wait test arms one row of the first token without its copy
      if (issued + 1 != p.withhold_row1) {
        if (p.keep_src0)
          bulk_copy_g2s_hint(ring + slot * (uint32_t)p.row_bytes, g, (uint32_t)p.row_bytes, full,
                             (j == 0 || j >= real_rows) ? keep : stream);
        else
          bulk_copy_g2s(ring + slot * (uint32_t)p.row_bytes, g, (uint32_t)p.row_bytes, full);
      }
      ++issued;
      if (++slot == (uint32_t)nslots) {
        slot = 0;
        ++lap;
      }
    }
  }
  if (!waited) {
    pdl_wait();
    pdl_trigger();
  }
  if (!ok) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
  ring_drain(sh.full, nslots, issued, p.withhold_row1);
}

// Launch of the multi-group kernel (aggregate_multi.cu).
cudaError_t launch_ring_multi(const RingParams& rp, int vpt, bool fused, bool exact, bool in_bf16, bool out_bf16,
                              int grid, int smem, cudaStream_t stream);

// The ring kernel for bf16 rows of d = 7168 with the source count fixed at
// compile time (ring_fixed_s.cu; fused: ring_fixed_s_fused.cu with a
// previous partial sum, ring_fixed_s_fused_noprev.cu without); rp.S in 1..9.
cudaError_t launch_ring_fixed_s(const RingParams& rp, int grid, int smem, cudaStream_t stream);
cudaError_t launch_ring_fixed_s_fused_prev(const RingParams& rp, int grid, int smem, cudaStream_t stream);
cudaError_t launch_ring_fixed_s_fused_noprev(const RingParams& rp, int grid, int smem, cudaStream_t stream);

// Split-d cluster variant for few tokens (aggregate_split.cu): the cluster
// size to use for T tokens (0 = none) and its launch.  Off unless the
// environment sets ATTNRES_SPLIT=1.
bool split_enabled();
int split_cluster_size(long long T, int sm_count, long long nvec);
cudaError_t launch_ring_split(const RingParams& rp_full, int C, bool fused, bool in_bf16, bool out_bf16,
                              int sm_count, int max_smem, cudaStream_t stream);

// Barrier set-up by thread 0 (the caller synchronises the CTA afterwards).
__device__ __forceinline__ void ring_init(const RingParams& p, RingShared& sh) {
  if (threadIdx.x == 0) {
    for (int k = 0; k < p.nslots; ++k) {
      mbar_init(smem_addr(&sh.full[k]), 1);
      mbar_init(smem_addr(&sh.empty[k]), kRingConsumerWarps);
    }
    sh.abort_flag[0] = 0;
    sh.abort_flag[1] = 0;
    sh.wait_ns = p.wait_ns;
    mbar_fence_init();
  }
}

}  // namespace attnres
