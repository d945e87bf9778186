// The hot-path ring kernel (agg_ring_kernel) and its launcher, shared by
// aggregate.cu (source count read at run time) and the translation units
// that instantiate it once per fixed source count (ring_fixed_s.cu,
// ring_fixed_s_fused.cu: bf16 rows of d = 7168, 1 <= S <= 9).  The
// arithmetic and the ring protocol are described at the top of aggregate.cu.
#pragma once

#include <atomic>
#include <math.h>

#include "attnres.h"
#include "device_common.cuh"
#include "launch.h"
#include "ring_common.cuh"

namespace attnres {

template <typename Tin, typename Tout, int VPT, bool FUSED, bool EXACT, int SC, int PREV = 0>
__global__ void __launch_bounds__(kRingThreads, 1) agg_ring_kernel(const __grid_constant__ RingParams p) {
  // EXACT: the row holds exactly VPT * kRingConsumers vectors, so every
  // consumer thread owns VPT of them and no bounds test is needed.
  // SC: the source count when fixed at compile time (0: p.S at run time);
  // with it the per-source guards fold away and the compiler schedules the
  // whole token as one block.
  // PREV (fused kernels): whether the fused source adds a previous partial
  // sum, fixed at compile time (1: no, 2: yes) or read from p (0).  Fixed, it
  // keeps the fused S = 9 kernel from spilling.
  constexpr int EPV = Vec<Tin>::kElems;
  // kEarlyRs: the first reduce-scatter level is taken per source during the
  // first pass (one partial live per source instead of two).  That keeps the
  // fused kernels (more live state) from spilling; the unfused ones are
  // faster without it at S = 9.
  constexpr bool kEarlyRs = FUSED;
  const bool has_prev = PREV == 0 ? p.fuse_prev != nullptr : PREV == 2;
  extern __shared__ __align__(128) unsigned char smem[];
  RingShared& sh = *reinterpret_cast<RingShared*>(smem);
  const uint32_t ring = smem_addr(smem) + kRingHeaderBytes;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nslots = p.nslots;
  const long long T = p.T;
  ring_init(p, sh);
  __syncthreads();

  if (warp == kRingConsumerWarps) {
    // the producer waits for the previous kernel itself (early loads)
    if (lane == 0) ring_produce(p, sh, ring);
    pdl_wait();
    pdl_trigger();
    return;
  }
  pdl_wait();  // everything below may read or overwrite what the previous kernel used
  pdl_trigger();

  // ------------------------------------------------------------ consumers --
  constexpr int NP = EPV / 2;  // packed fp32 pairs per 16-byte vector
  uint64_t wp[VPT][NP];        // this thread's channels of w, as pairs
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * kRingConsumers;
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const bool in = EXACT || v < p.nvec;
      wp[k][j] = f2_pack(in ? __ldg(p.w + v * EPV + 2 * j) : 0.f, in ? __ldg(p.w + v * EPV + 2 * j + 1) : 0.f);
    }
  }

  const int S = SC ? SC : p.S;
  uint32_t slot = 0, lap = 0;
  bool ok = true;

  // take this thread's vectors of the next landed row, then release the slot
  auto consume = [&](uint4* dst) {
    if (ok && !mbar_wait_bounded_sh(smem_addr(&sh.full[slot]), lap & 1u, &sh.wait_ns)) ok = false;
    const uint32_t base = ring + slot * (uint32_t)p.row_bytes;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * kRingConsumers;
      // after a failed wait the slot holds stale data: harmless, the token is abandoned
      dst[k] = (EXACT || v < p.nvec) ? ld_shared_v4(base + (uint32_t)v * 16u) : make_uint4(0, 0, 0, 0);
    }
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

  // NR: the sources the reductions carry (the fixed count, else 9).  A
  // token's partials are [dot(w, h_0..h_NR-1), sum(h_0^2)..sum(h_NR-1^2)],
  // summed over the warp by a reduce-scatter of 2 NR values (20 shuffles at
  // NR = 9, 6 at NR = 2).
  constexpr int NR = SC ? SC : kRingSmax;
  int iter = 0;
  for (long long t = blockIdx.x; t < T; t += gridDim.x, ++iter) {
    const int buf = iter & 1;
    volatile int* abort_flag = &sh.abort_flag[buf];
    uint4 x[kRingSmax][VPT];
    // With kEarlyRs, per source, this thread's dot and sum of squares enter
    // the first level of the warp reduce-scatter at once: lanes with bit 4
    // clear keep the dot products, the others the sums of squares, each
    // adding its partner's (lane ^ 16).
    const bool upper16 = (lane & 16) != 0;
    float part[kEarlyRs ? NR : 2 * NR];
#pragma unroll
    for (int s = 0; s < (kEarlyRs ? NR : 2 * NR); ++s) part[s] = 0.f;
#pragma unroll
    for (int s = 0; s < NR; ++s) {
      if (s < S) {
        if (!FUSED || s < p.n_stored) {
          consume(x[s]);
        } else {
          // the fused source: round(prev + F), stored as the new partial / b_n
          uint4 pv[VPT], fv[VPT];
          if (has_prev) consume(pv);
          consume(fv);
          char* drow = p.fuse_dst + t * (long long)p.row_bytes;
#pragma unroll
          for (int k = 0; k < VPT; ++k) {
            const int v = tid + k * kRingConsumers;
            if (EXACT || v < p.nvec) {
              float f[EPV];
              Vec<Tin>::unpack(fv[k], f);
              if (has_prev) {
                float q[EPV];
                Vec<Tin>::unpack(pv[k], q);
#pragma unroll
                for (int e = 0; e < EPV; ++e) f[e] = q[e] + f[e];
              }
              if (!ok) {
#pragma unroll
                for (int e = 0; e < EPV; ++e) f[e] = __int_as_float(0x7fc00000);
              }
              x[s][k] = Vec<Tin>::pack(f);  // one rounding to the storage type
              *reinterpret_cast<uint4*>(drow + (size_t)v * 16) = x[s][k];
            } else {
              x[s][k] = make_uint4(0, 0, 0, 0);
            }
          }
        }
        // two packed accumulators each (four partial sums) to keep the
        // dependent FMA chains short
        uint64_t dot2[2] = {0, 0}, ss2[2] = {0, 0};
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          uint64_t h[NP];
          Vec<Tin>::pairs(x[s][k], h);
#pragma unroll
          for (int j = 0; j < NP; ++j) {
            dot2[j & 1] = f2_fma(wp[k][j], h[j], dot2[j & 1]);
            ss2[j & 1] = f2_fma(h[j], h[j], ss2[j & 1]);
          }
        }
        const float dot = f2_hsum(dot2[0]) + f2_hsum(dot2[1]);
        const float ss = f2_hsum(ss2[0]) + f2_hsum(ss2[1]);
        if constexpr (kEarlyRs) {
          part[s] = (upper16 ? ss : dot) + __shfl_xor_sync(0xffffffffu, upper16 ? dot : ss, 16);
        } else {
          part[s] = dot;
          part[NR + s] = ss;
        }
      }
    }

    // ---- warp totals (reduce-scatter), then one CTA-wide step through smem;
    // value index i < NR is dot(w, h_i), NR + i is sum(h_i^2), stored at [2i]
    // and [2i + 1]
    if constexpr (kEarlyRs) reduce_scatter_after_first<2 * NR>(part, lane);
    else reduce_scatter<2 * NR>(part, lane);
    const int rs_idx = rs_lane_index<2 * NR>(lane);  // value whose warp total this lane holds (-1: none)
    if (rs_idx >= 0) {
      const int src = rs_idx < NR ? rs_idx : rs_idx - NR;
      if (src < S) sh.red[buf][warp][rs_idx < NR ? 2 * rs_idx : 2 * src + 1] = part[0];
    }
    const bool warp_failed = __any_sync(0xffffffffu, !ok);
    if (lane == 0 && warp_failed) *abort_flag = 1;
    named_barrier_sync(kRingBarrierId, kRingConsumers);

    // ---- logits and the depth softmax, computed by every warp (lane 2s
    // holds source s); all warps sum in the same order, so agree bit for bit
    const bool abort = *abort_flag != 0;
    float tot = 0.f;
    if (lane < 2 * S) {
#pragma unroll
      for (int w = 0; w < kRingConsumerWarps; ++w) tot += sh.red[buf][w][lane];
    }
    const float sumsq = __shfl_down_sync(0xffffffffu, tot, 1);
    const bool is_src = lane < 2 * S && (lane & 1) == 0;
    // fast reciprocal square root, exponential and division: each within a
    // few fp32 ulps, far inside the 1e-5 weight tolerance
    const float z = is_src ? tot * rsqrtf(fmaf(sumsq, p.inv_d, p.eps)) : -INFINITY;
    const float m = warp_max(z);
    const float e = is_src ? __expf(z - m) : 0.f;
    const float esum = warp_sum(e);
    float a = abort ? __int_as_float(0x7fc00000) : __fdividef(e, esum);
    if (warp == 0 && is_src && p.out_a) p.out_a[t * S + (lane >> 1)] = a;
    // ---- r = sum_s a_s h_s from the registers
    uint64_t acc[VPT][NP];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
#pragma unroll
      for (int j = 0; j < NP; ++j) acc[k][j] = 0;
    }
    {
      if constexpr (SC != 0) {
        // With a fixed source count the compiler would otherwise keep the
        // first pass's unpacked fp32 values alive across the barrier (twice
        // the registers, spilled); the empty asm makes it unpack the packed
        // registers again instead.
#pragma unroll
        for (int s = 0; s < NR; ++s) {
#pragma unroll
          for (int k = 0; k < VPT; ++k)
            asm volatile("" : "+r"(x[s][k].x), "+r"(x[s][k].y), "+r"(x[s][k].z), "+r"(x[s][k].w));
        }
      }
      uint64_t a2[NR];
#pragma unroll
      for (int s = 0; s < NR; ++s) {
        const float as = __shfl_sync(0xffffffffu, a, 2 * s);
        a2[s] = f2_pack(as, as);
      }
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
#pragma unroll
        for (int s = 0; s < NR; ++s) {
          if (s < S) {
            uint64_t h[NP];
            Vec<Tin>::pairs(x[s][k], h);
#pragma unroll
            for (int j = 0; j < NP; ++j) acc[k][j] = f2_fma(a2[s], h[j], acc[k][j]);
          }
        }
      }
    }
    char* orow = p.out_r + t * (long long)p.out_row_bytes;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * kRingConsumers;
      if (EXACT || v < p.nvec) {
        float r[EPV];
#pragma unroll
        for (int j = 0; j < NP; ++j) f2_unpack(acc[k][j], r[2 * j], r[2 * j + 1]);
        if (abort) {
#pragma unroll
          for (int e2 = 0; e2 < EPV; ++e2) r[e2] = __int_as_float(0x7fc00000);
        }
        store_out<Tout, EPV>(orow, v, r);
      }
    }
    if (abort) {
      if (tid == 0) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
      break;
    }
  }
}

template <typename Tin, typename Tout, int VPT, bool FUSED, bool EXACT, int SC = 0, int PREV = 0>
static cudaError_t launch_ring_t(const RingParams& rp, int grid, int smem, cudaStream_t stream) {
  static SmemOptIn optin;  // the large shared-memory opt-in, per device and context
  auto kern = agg_ring_kernel<Tin, Tout, VPT, FUSED, EXACT, SC, PREV>;
  cudaError_t e = optin.ensure(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  e = launch_kernel(kern, dim3(grid), dim3(kRingThreads), (size_t)smem, stream, rp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace attnres
