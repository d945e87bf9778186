// Depth-wise attention over MORE than 9 sources per token (Full AttnRes:
// block size 1 gives layer l its l sources, up to 94 for 93 layers; Kimi K3
// chaptered tutorial, ch. 4.2 Eq. 8-9).  Same ring design as the 9-source
// kernel in ring_kernel.cuh (persistent CTA per SM, TMA bulk copies of source
// rows into a shared-memory ring, consumer threads owning fixed 16-byte
// vectors), but a token's sources are taken in groups of up to 9 and folded
// into the output with an online softmax (tutorial, ch. 4.4: a running
// maximum m and running sum l, partial results rescaled when m grows):
//
//   for each group g:  z_s = w . RMSNorm(h_s)            (s in g)
//                      m' = max(m, max_s z_s),  c = exp(m - m')
//                      l  = l c + sum_s exp(z_s - m')
//                      acc = acc c + sum_s exp(z_s - m') h_s
//                      m  = m'
//   r = acc / l;   a_s = exp(z_s - m) / l   (logits kept in shared memory)
//
// Every source byte is still read from HBM once; each group costs one
// cross-warp reduction step (one named barrier).  A token's source list is
// padded to a whole number of groups; a padding position's logit is -inf
// (weight exactly 0), so every group has the compile-time size and the
// per-source guards fold away.  In a plain aggregation the padding rows are
// re-reads of the token's source 0 row (L2-resident by then).  In a fused
// step the token's last group, which holds the formed source (prev + F),
// is compiled with per-position checks, and its padding positions take no
// ring slot and no load: their rows are zero.
#include <atomic>
#include <math.h>
#include <type_traits>

#include "ring_common.cuh"

namespace attnres {

// GS: sources per group (<= 9); smaller groups leave registers for the
// running accumulator where a 16-byte vector holds 8 bf16 values.
template <typename Tin, int VPT>
struct MultiGroup {
  static constexpr int kSize = (sizeof(Tin) == 2 && VPT == 2) ? 6 : kRingSmax;
};

template <typename Tin, typename Tout, int VPT, bool FUSED, bool EXACT>
__global__ void __launch_bounds__(kRingThreads, 1) agg_ring_multi_kernel(const __grid_constant__ RingParams p) {
  constexpr int GS = MultiGroup<Tin, VPT>::kSize;
  constexpr int EPV = Vec<Tin>::kElems;
  constexpr int NP = EPV / 2;
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
  pdl_wait();  // everything below may read what the previous kernel wrote
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done

  if (warp == kRingConsumerWarps) {
    if (lane == 0) ring_produce(p, sh, ring);
    return;
  }

  // ------------------------------------------------------------ consumers --
  uint64_t wp[VPT][NP];  // this thread's channels of w, as pairs
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * kRingConsumers;
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const bool in = EXACT || v < p.nvec;
      wp[k][j] = f2_pack(in ? __ldg(p.w + v * EPV + 2 * j) : 0.f, in ? __ldg(p.w + v * EPV + 2 * j + 1) : 0.f);
    }
  }

  const int S = p.S;
  const int S_pad = (S + GS - 1) / GS * GS;  // a whole number of groups of GS (padding weighs 0)
  uint32_t slot = 0, lap = 0;
  bool ok = true;

  // take this thread's vectors of the next landed row, then release the slot
  auto consume = [&](uint4* dst) {
    if (ok && !mbar_wait_bounded(smem_addr(&sh.full[slot]), lap & 1u, p.wait_ns)) ok = false;
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

  // the value of a group's [dot_0, ss_0, dot_1, ss_1, ...] partials whose
  // warp total this lane holds after the reduce-scatter (-1: none)
  const int rs_idx = rs_lane_index<2 * GS>(lane);
  int iter = 0;  // groups processed by this CTA (selects the reduction buffer)
  bool abort = false;
  for (long long t = blockIdx.x; t < T && !abort; t += gridDim.x) {
    float m = -INFINITY, l = 0.f;
    uint64_t acc[VPT][NP];
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
      for (int j = 0; j < NP; ++j) acc[k][j] = 0;

    for (int g0 = 0; g0 < S_pad; g0 += GS, ++iter) {
      const int buf = iter & 1;
      volatile int* abort_flag = &sh.abort_flag[buf];
      uint4 x[GS][VPT];
      float part[2 * GS];  // every entry is set below
      // The group's rows and their partial dots.  Stored sources and a plain
      // aggregation's padding are single rows; a fused step's source (index
      // n_stored = S - 1) is formed from prev and F, and its padding
      // positions (index >= S) are zero rows with zero partials, loaded from
      // nowhere.  Only a fused step's last group is compiled with those
      // checks: the other groups stay straight-line code, so one row's loads
      // overlap the previous row's arithmetic.
      auto load_group = [&](auto last_group) {
        constexpr bool LAST = decltype(last_group)::value;
#pragma unroll
        for (int s = 0; s < GS; ++s) {
          if (LAST && g0 + s >= S) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) x[s][k] = make_uint4(0, 0, 0, 0);
            part[2 * s] = 0.f;
            part[2 * s + 1] = 0.f;
            continue;
          }
          if (!(LAST && FUSED) || g0 + s != p.n_stored) {
            consume(x[s]);
          } else {
            // the fused source (the token's last): round(prev + F), stored as
            // the new partial sum / block representation
            uint4 pv[VPT], fv[VPT];
            if (p.fuse_prev) consume(pv);
            consume(fv);
            char* drow = p.fuse_dst + t * (long long)p.row_bytes;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
              const int v = tid + k * kRingConsumers;
              if (EXACT || v < p.nvec) {
                float f[EPV];
                Vec<Tin>::unpack(fv[k], f);
                if (p.fuse_prev) {
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
          part[2 * s] = f2_hsum(dot2[0]) + f2_hsum(dot2[1]);
          part[2 * s + 1] = f2_hsum(ss2[0]) + f2_hsum(ss2[1]);
        }
      };
      if (FUSED && g0 + GS == S_pad)
        load_group(std::true_type{});
      else
        load_group(std::false_type{});

      // ---- warp totals (a reduce-scatter over the group's 2 GS partials:
      // 13 shuffles for GS = 6), then one CTA-wide step
      reduce_scatter<2 * GS>(part, lane);
      if (rs_idx >= 0) sh.red[buf][warp][rs_idx] = part[0];
      const bool warp_failed = __any_sync(0xffffffffu, !ok);
      if (lane == 0 && warp_failed) *abort_flag = 1;
      named_barrier_sync(kRingBarrierId, kRingConsumers);

      // ---- this group's logits, folded into the running softmax (lane 2s
      // holds source g0+s; all warps agree bit for bit)
      abort = *abort_flag != 0;
      float tot = 0.f;
      if (lane < 2 * GS) {
#pragma unroll
        for (int w = 0; w < kRingConsumerWarps; ++w) tot += sh.red[buf][w][lane];
      }
      const float sumsq = __shfl_down_sync(0xffffffffu, tot, 1);
      // padding sources (index >= S) get a logit of -inf: weight exactly 0
      const bool is_src = lane < 2 * GS && (lane & 1) == 0 && g0 + (lane >> 1) < S;
      // fast reciprocal square root and exponential: a few fp32 ulps, far
      // inside the 1e-5 weight tolerance
      const float z = is_src ? tot * rsqrtf(fmaf(sumsq, p.inv_d, p.eps)) : -INFINITY;
      const float m_new = fmaxf(m, warp_max(z));
      const float c = __expf(m - m_new);  // 0 for the first group (m = -inf)
      const float e = is_src ? __expf(z - m_new) : 0.f;
      l = l * c + warp_sum(e);
      if (warp == 0 && is_src) sh.zbuf[g0 + (lane >> 1)] = z;
      m = m_new;
      // re-materialise the packed sources so the compiler does not keep the
      // first pass's unpacked values across the barrier (that spills)
#pragma unroll
      for (int s = 0; s < GS; ++s) {
#pragma unroll
        for (int k = 0; k < VPT; ++k)
          asm volatile("" : "+r"(x[s][k].x), "+r"(x[s][k].y), "+r"(x[s][k].z), "+r"(x[s][k].w));
      }
      const uint64_t c2 = f2_pack(c, c);
      uint64_t e2[GS];
#pragma unroll
      for (int s = 0; s < GS; ++s) {
        const float es = __shfl_sync(0xffffffffu, e, 2 * s);
        e2[s] = f2_pack(es, es);
      }
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = tid + k * kRingConsumers;
        if (EXACT || v < p.nvec) {
#pragma unroll
          for (int j = 0; j < NP; ++j) acc[k][j] = f2_fma(acc[k][j], c2, 0);
#pragma unroll
          for (int s = 0; s < GS; ++s) {
            uint64_t h[NP];
            Vec<Tin>::pairs(x[s][k], h);
#pragma unroll
            for (int j = 0; j < NP; ++j) acc[k][j] = f2_fma(e2[s], h[j], acc[k][j]);
          }
        }
      }
      if (abort) break;
    }

    // ---- r = acc / l, and the weights exp(z_s - m) / l
    const float inv = __fdividef(1.0f, l);
    const uint64_t inv2 = f2_pack(inv, inv);
    char* orow = p.out_r + t * (long long)p.out_row_bytes;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * kRingConsumers;
      if (EXACT || v < p.nvec) {
        float r[EPV];
#pragma unroll
        for (int j = 0; j < NP; ++j) f2_unpack(f2_fma(acc[k][j], inv2, 0), r[2 * j], r[2 * j + 1]);
        if (abort) {
#pragma unroll
          for (int e2 = 0; e2 < EPV; ++e2) r[e2] = __int_as_float(0x7fc00000);
        }
        store_out<Tout, EPV>(orow, v, r);
      }
    }
    if (warp == 0 && p.out_a) {
      __syncwarp();
      for (int s = lane; s < S; s += 32)
        p.out_a[t * S + s] = abort ? __int_as_float(0x7fc00000) : __expf(sh.zbuf[s] - m) * inv;
      __syncwarp();
    }
    if (abort && tid == 0) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
  }
}

template <typename Tin, typename Tout, int VPT, bool FUSED, bool EXACT>
static cudaError_t launch_multi_t(const RingParams& rp, int grid, int smem, cudaStream_t stream) {
  static SmemOptIn optin;  // the large shared-memory opt-in, per device and context
  auto kern = agg_ring_multi_kernel<Tin, Tout, VPT, FUSED, EXACT>;
  cudaError_t e = optin.ensure(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  // a plain aggregation's padding to a whole number of groups: re-reads of
  // source 0 (a fused step pads without rows)
  constexpr int GS = MultiGroup<Tin, VPT>::kSize;
  RingParams padded = rp;
  padded.pad_rows = FUSED ? 0 : (GS - rp.S % GS) % GS;
  e = launch_kernel(kern, dim3(grid), dim3(kRingThreads), (size_t)smem, stream, padded);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename Tin, typename Tout>
static cudaError_t launch_multi_vpt(const RingParams& rp, int vpt, bool fused, bool exact, int grid, int smem,
                                    cudaStream_t stream) {
  if (vpt == 1) {
    return fused ? launch_multi_t<Tin, Tout, 1, true, false>(rp, grid, smem, stream)
                 : launch_multi_t<Tin, Tout, 1, false, false>(rp, grid, smem, stream);
  }
  if (exact) {
    return fused ? launch_multi_t<Tin, Tout, 2, true, true>(rp, grid, smem, stream)
                 : launch_multi_t<Tin, Tout, 2, false, true>(rp, grid, smem, stream);
  }
  return fused ? launch_multi_t<Tin, Tout, 2, true, false>(rp, grid, smem, stream)
               : launch_multi_t<Tin, Tout, 2, false, false>(rp, grid, smem, stream);
}

cudaError_t launch_ring_multi(const RingParams& rp, int vpt, bool fused, bool exact, bool in_bf16, bool out_bf16,
                              int grid, int smem, cudaStream_t stream) {
  if (in_bf16) {
    return out_bf16 ? launch_multi_vpt<bf16_t, bf16_t>(rp, vpt, fused, exact, grid, smem, stream)
                    : launch_multi_vpt<bf16_t, float>(rp, vpt, fused, exact, grid, smem, stream);
  }
  return out_bf16 ? launch_multi_vpt<float, bf16_t>(rp, vpt, fused, exact, grid, smem, stream)
                  : launch_multi_vpt<float, float>(rp, vpt, fused, exact, grid, smem, stream);
}

}  // namespace attnres
