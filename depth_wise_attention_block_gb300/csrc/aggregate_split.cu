// Depth-wise attention for few tokens (decode: T = 64 leaves most SMs idle
// with one CTA per token), an opt-in variant: a thread-block cluster of C
// CTAs shares each token, every CTA streaming and owning one channel slice
// of every source row.  The math is that of agg_ring_kernel
// (ring_kernel.cuh); per token each CTA reduces its slice's dot(w, h_s) and
// sum(h_s^2) partials as usual, then the C slice totals are exchanged
// through distributed shared memory: lane 0 of warp 0 stores its CTA's 2S
// totals into every CTA's exchange buffer of the cluster and arrives
// (release, cluster scope) on each CTA's exchange mbarrier (C arrivals
// complete it, its own included); every consumer warp waits on its own CTA's
// mbarrier and sums the C contributions in rank order, so all CTAs form
// bit-identical logits and weights, then writes its slice of r.  The
// exchange buffers and mbarriers are double-buffered: a peer overwrites
// buffer b only after this CTA's arrival for the next token, which comes
// after all of its warps have read buffer b.  A cluster barrier after the
// set-up and another before exit keep every CTA alive while a peer may still
// write into it.  No multicast.
#include <atomic>
#include <math.h>
#include <stdlib.h>

#include "ring_common.cuh"

namespace attnres {

constexpr int kSplitMaxC = 8;

struct SplitShared {
  RingShared ring_hdr;  // full / empty barriers, per-warp reduction buffers, abort flags
  uint64_t xbar[2];     // exchange completion, one per token parity
  float xbuf[2][kSplitMaxC][2 * kRingSmax];
};
constexpr int kSplitHeaderBytes = (int)((sizeof(SplitShared) + 127) / 128 * 128);

struct SplitParams {
  RingParams rp;         // rp.row_bytes = slice bytes copied per row, rp.nvec = vectors per slice
  long long row_stride;  // bytes between consecutive tokens' rows (the full row)
  long long out_stride;  // bytes between consecutive tokens' output rows
  int C;                 // CTAs per cluster
  int out_slice_bytes;   // bytes of one CTA's slice of an output row
};

// Producer: this CTA's slice of every row of the cluster's tokens.
__device__ __forceinline__ void split_produce(const SplitParams& sp, RingShared& sh, uint32_t ring, uint32_t rank,
                                              long long cluster, long long nclusters) {
  const RingParams& p = sp.rp;
  const int nslots = p.nslots;
  const bool fused = p.fuse_F != nullptr;
  const int rows = p.n_stored + (fused ? (p.fuse_prev ? 2 : 1) : 0);
  const long long slice_off = (long long)rank * p.row_bytes;
  uint32_t slot = 0, lap = 0;
  long long issued = 0;
  bool ok = true;
  for (long long t = cluster; t < p.T && ok; t += nclusters) {
    const long long off = t * sp.row_stride + slice_off;
    for (int j = 0; j < rows; ++j) {
      const char* g;
      if (j < p.n_stored) g = p.src[j] + off;
      else if (p.fuse_prev && j == p.n_stored) g = p.fuse_prev + off;
      else g = p.fuse_F + off;
      if (!mbar_wait_bounded(smem_addr(&sh.empty[slot]), (lap & 1u) ^ 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      const uint32_t full = smem_addr(&sh.full[slot]);
      mbar_arrive_expect_tx(full, (uint32_t)p.row_bytes);
      // the bounded-wait test arms one row of the first token without its copy
      if (issued + 1 != p.withhold_row1)
        bulk_copy_g2s(ring + slot * (uint32_t)p.row_bytes, g, (uint32_t)p.row_bytes, full);
      ++issued;
      if (++slot == (uint32_t)nslots) {
        slot = 0;
        ++lap;
      }
    }
  }
  if (!ok) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
  ring_drain(sh.full, nslots, issued, p.withhold_row1);
}

template <typename Tin, typename Tout, bool FUSED>
__global__ void __launch_bounds__(kRingThreads, 1) agg_split_kernel(const __grid_constant__ SplitParams sp) {
  const RingParams& p = sp.rp;
  constexpr int EPV = Vec<Tin>::kElems;
  constexpr int NP = EPV / 2;
  extern __shared__ __align__(128) unsigned char smem[];
  SplitShared& xs = *reinterpret_cast<SplitShared*>(smem);
  RingShared& sh = xs.ring_hdr;
  const uint32_t ring = smem_addr(smem) + kSplitHeaderBytes;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int C = sp.C;
  const uint32_t rank = cluster_ctarank();
  const long long cluster = blockIdx.x / C;
  const long long nclusters = gridDim.x / C;
  ring_init(p, sh);
  if (tid == 0) {
    mbar_init(smem_addr(&xs.xbar[0]), C);
    mbar_init(smem_addr(&xs.xbar[1]), C);
    mbar_fence_init();
  }
  __syncthreads();  // this CTA's ring barriers exist
  // every CTA's exchange barriers exist before any peer touches them: the
  // consumers wait for the cluster barrier now, the producer only after its
  // copies are issued
  cluster_arrive();
  pdl_wait();
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done

  if (warp == kRingConsumerWarps) {
    if (lane == 0) split_produce(sp, sh, ring, rank, cluster, nclusters);
    __syncwarp();
    cluster_wait();
    cluster_sync_all();
    return;
  }
  cluster_wait();

  // ------------------------------------------------------------ consumers --
  const int nvec = p.nvec;  // this CTA's vectors per row (<= 448: one per thread)
  const int v = tid;
  const bool mine = v < nvec;
  const long long ch0 = (long long)rank * nvec * EPV;  // first channel of the slice
  uint64_t wp[NP];
#pragma unroll
  for (int j = 0; j < NP; ++j)
    wp[j] = f2_pack(mine ? __ldg(p.w + ch0 + v * EPV + 2 * j) : 0.f, mine ? __ldg(p.w + ch0 + v * EPV + 2 * j + 1) : 0.f);

  const int S = p.S;
  const int nslots = p.nslots;
  uint32_t slot = 0, lap = 0;
  bool ok = true;
  auto consume = [&](uint4& dst) {
    if (ok && !mbar_wait_bounded(smem_addr(&sh.full[slot]), lap & 1u, p.wait_ns)) ok = false;
    const uint32_t base = ring + slot * (uint32_t)p.row_bytes;
    dst = mine ? ld_shared_v4(base + (uint32_t)v * 16u) : make_uint4(0, 0, 0, 0);
    // Lane 0 releases the slot only while its own waits have all succeeded:
    // then this phase completed and its copy landed.  After a wait ran out
    // the copy may still be in flight, and the slot must not be refilled
    // under it (the producer then runs out of slots, stops and drains).
    __syncwarp();
    if (lane == 0 && ok) mbar_arrive(smem_addr(&sh.empty[slot]));
    if (++slot == (uint32_t)nslots) {
      slot = 0;
      ++lap;
    }
  };

  int iter = 0;
  bool abort = false;
  for (long long t = cluster; t < p.T && !abort; t += nclusters, ++iter) {
    const int buf = iter & 1;
    volatile int* abort_flag = &sh.abort_flag[buf];
    uint4 x[kRingSmax];
    float part[2 * kRingSmax];
#pragma unroll
    for (int s = 0; s < kRingSmax; ++s) {
      part[2 * s] = 0.f;
      part[2 * s + 1] = 0.f;
      if (s < S) {
        if (!FUSED || s < p.n_stored) {
          consume(x[s]);
        } else {
          uint4 pv = make_uint4(0, 0, 0, 0), fv;
          if (p.fuse_prev) consume(pv);
          consume(fv);
          x[s] = make_uint4(0, 0, 0, 0);
          if (mine) {
            float f[EPV];
            Vec<Tin>::unpack(fv, f);
            if (p.fuse_prev) {
              float q[EPV];
              Vec<Tin>::unpack(pv, q);
#pragma unroll
              for (int e = 0; e < EPV; ++e) f[e] = q[e] + f[e];
            }
            if (!ok) {
#pragma unroll
              for (int e = 0; e < EPV; ++e) f[e] = __int_as_float(0x7fc00000);
            }
            x[s] = Vec<Tin>::pack(f);  // one rounding to the storage type
            char* drow = p.fuse_dst + t * sp.row_stride + (long long)rank * p.row_bytes;
            *reinterpret_cast<uint4*>(drow + (size_t)v * 16) = x[s];
          }
        }
        uint64_t dot2 = 0, ss2 = 0;
        uint64_t h[NP];
        Vec<Tin>::pairs(x[s], h);
#pragma unroll
        for (int j = 0; j < NP; ++j) {
          dot2 = f2_fma(wp[j], h[j], dot2);
          ss2 = f2_fma(h[j], h[j], ss2);
        }
        part[2 * s] = f2_hsum(dot2);
        part[2 * s + 1] = f2_hsum(ss2);
      }
    }

    // ---- this CTA's slice totals
    reduce_scatter18(part, lane);
    if ((kRsValidLanes >> lane) & 1u) {
      const int idx = rs_index(lane);
      if (idx < 2 * S) sh.red[buf][warp][idx] = part[0];
    }
    const bool warp_failed = __any_sync(0xffffffffu, !ok);
    if (lane == 0 && warp_failed) *abort_flag = 1;
    named_barrier_sync(kRingBarrierId, kRingConsumers);

    // the CTA-uniform exit test: every warp reads the flag after the barrier
    abort = *abort_flag != 0;
    if (abort) {
      if (mine) {
        float r[EPV];
#pragma unroll
        for (int e2 = 0; e2 < EPV; ++e2) r[e2] = __int_as_float(0x7fc00000);
        store_out<Tout, EPV>(p.out_r + t * sp.out_stride + (long long)rank * sp.out_slice_bytes, v, r);
      }
      if (rank == 0 && p.out_a && tid < S) p.out_a[t * S + tid] = __int_as_float(0x7fc00000);
      if (tid == 0) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
      break;
    }

    // ---- exchange across the cluster: lane 0 of warp 0 stores this CTA's
    // 2S slice totals into every CTA's buffer (its own included), then
    // arrives on every CTA's exchange barrier (release: its stores first)
    const uint32_t xbar = smem_addr(&xs.xbar[buf]);
    if (warp == 0) {
      float mytot = 0.f;
      if (lane < 2 * S) {
#pragma unroll
        for (int w = 0; w < kRingConsumerWarps; ++w) mytot += sh.red[buf][w][lane];
      }
      float vals[2 * kRingSmax];
#pragma unroll
      for (int j = 0; j < 2 * kRingSmax; ++j) vals[j] = __shfl_sync(0xffffffffu, mytot, j);
      if (lane == 0) {
        const uint32_t base = smem_addr(&xs.xbuf[buf][rank][0]);
        for (int c = 0; c < C; ++c) {
          const uint32_t remote = map_shared_rank(base, (uint32_t)c);
#pragma unroll
          for (int j = 0; j < 2 * kRingSmax; ++j)
            if (j < 2 * S) st_shared_cluster_f32(remote + 4u * (uint32_t)j, vals[j]);
        }
        for (int c = 0; c < C; ++c) mbar_arrive_cluster(map_shared_rank(xbar, (uint32_t)c));
      }
      __syncwarp();
    }
    // a wait that runs out poisons this token here and, through `ok`, the
    // abort flag at the next token's barrier
    if (!mbar_wait_cluster_bounded(xbar, (uint32_t)((iter >> 1) & 1))) ok = false;
    const bool token_ok = __all_sync(0xffffffffu, ok);

    float tot = 0.f;
    if (lane < 2 * S) {
      for (int c = 0; c < C; ++c) tot += xs.xbuf[buf][c][lane];
    }
    const float sumsq = __shfl_down_sync(0xffffffffu, tot, 1);
    const bool is_src = lane < 2 * S && (lane & 1) == 0;
    // fast reciprocal square root, exponential and division: a few fp32 ulps
    const float z = is_src ? tot * rsqrtf(fmaf(sumsq, p.inv_d, p.eps)) : -INFINITY;
    const float m = warp_max(z);
    const float e = is_src ? __expf(z - m) : 0.f;
    const float esum = warp_sum(e);
    const bool bad = !token_ok;
    const float a = bad ? __int_as_float(0x7fc00000) : __fdividef(e, esum);
    if (rank == 0 && warp == 0 && is_src && p.out_a) p.out_a[t * S + (lane >> 1)] = a;
    uint64_t a2[kRingSmax];
#pragma unroll
    for (int s = 0; s < kRingSmax; ++s) {
      const float as = __shfl_sync(0xffffffffu, a, 2 * s);
      a2[s] = f2_pack(as, as);
    }
    if (mine) {
      uint64_t acc[NP];
#pragma unroll
      for (int j = 0; j < NP; ++j) acc[j] = 0;
#pragma unroll
      for (int s = 0; s < kRingSmax; ++s) {
        if (s < S) {
          uint64_t h[NP];
          Vec<Tin>::pairs(x[s], h);
#pragma unroll
          for (int j = 0; j < NP; ++j) acc[j] = f2_fma(a2[s], h[j], acc[j]);
        }
      }
      float r[EPV];
#pragma unroll
      for (int j = 0; j < NP; ++j) f2_unpack(acc[j], r[2 * j], r[2 * j + 1]);
      if (bad) {
#pragma unroll
        for (int e2 = 0; e2 < EPV; ++e2) r[e2] = __int_as_float(0x7fc00000);
      }
      store_out<Tout, EPV>(p.out_r + t * sp.out_stride + (long long)rank * sp.out_slice_bytes, v, r);
    }
    if (bad && tid == 0) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
  }
  cluster_sync_all();  // no CTA leaves while a peer may still write into it
}

template <typename Tin, typename Tout, bool FUSED>
static cudaError_t launch_split_t(const SplitParams& sp, int grid, int smem, cudaStream_t stream) {
  static SmemOptIn optin;  // the large shared-memory opt-in, per device and context
  auto kern = agg_split_kernel<Tin, Tout, FUSED>;
  cudaError_t e = optin.ensure(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRingThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = sp.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kern, sp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Cluster size for T tokens (0 = do not split).  Every CTA keeps at least
// 64 vectors (1 KB of bf16) of each row, so the exchange stays small against
// the streaming.  Off unless ATTNRES_SPLIT=1: on GB300 at d = 7168 a launch
// over T <= 76 tokens is bound by fixed latency (about 5 us at S = 9 from
// T = 1 to 76 with one CTA per token), which the cluster barriers and the
// exchange add to rather than hide.
int split_cluster_size(long long T, int sm_count, long long nvec) {
  if (!split_enabled()) return 0;
  for (int C : {8, 4, 2}) {
    if (nvec % C != 0 || nvec / C > kRingConsumers || nvec / C < 64) continue;
    if ((long long)C * T <= sm_count) return C;
  }
  return 0;
}

bool split_enabled() {
  static const bool on = [] {
    const char* v = getenv("ATTNRES_SPLIT");
    return v && v[0] && v[0] != '0';
  }();
  return on;
}

cudaError_t launch_ring_split(const RingParams& rp_full, int C, bool fused, bool in_bf16, bool out_bf16,
                              int sm_count, int max_smem, cudaStream_t stream) {
  SplitParams sp{};
  sp.rp = rp_full;
  sp.C = C;
  sp.row_stride = rp_full.row_bytes;
  sp.out_stride = rp_full.out_row_bytes;
  sp.rp.nvec = rp_full.nvec / C;
  sp.rp.row_bytes = rp_full.row_bytes / C;
  sp.out_slice_bytes = rp_full.out_row_bytes / C;
  int nslots = (max_smem - kSplitHeaderBytes) / sp.rp.row_bytes;
  if (nslots > kRingMaxSlots) nslots = kRingMaxSlots;
  if (nslots < 1) return cudaErrorInvalidValue;
  sp.rp.nslots = nslots;
  const int nclusters = (int)(rp_full.T * C <= sm_count ? rp_full.T : sm_count / C);
  const int grid = nclusters * C;
  const int smem = kSplitHeaderBytes + nslots * sp.rp.row_bytes;
  if (in_bf16) {
    if (out_bf16) return fused ? launch_split_t<bf16_t, bf16_t, true>(sp, grid, smem, stream)
                               : launch_split_t<bf16_t, bf16_t, false>(sp, grid, smem, stream);
    return fused ? launch_split_t<bf16_t, float, true>(sp, grid, smem, stream)
                 : launch_split_t<bf16_t, float, false>(sp, grid, smem, stream);
  }
  if (out_bf16) return fused ? launch_split_t<float, bf16_t, true>(sp, grid, smem, stream)
                             : launch_split_t<float, bf16_t, false>(sp, grid, smem, stream);
  return fused ? launch_split_t<float, float, true>(sp, grid, smem, stream)
               : launch_split_t<float, float, false>(sp, grid, smem, stream);
}

}  // namespace attnres
