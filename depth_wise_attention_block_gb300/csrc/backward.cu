// Backward of one layer of depth-wise attention, recomputing the forward
// (AttnRes runs under activation checkpointing in training: Kimi K3
// chaptered tutorial, ch. 4.6).  Per token, with rho_s = rms(h_s),
// z_s = (w . h_s) / rho_s, a = softmax(z), r = sum_s a_s h_s and the
// incoming gradient dr of r:
//
//   g_s   = dr . h_s,   gbar = sum_s a_s g_s,   dz_s = a_s (g_s - gbar)
//   alpha_s = dz_s / rho_s,   beta_s = alpha_s z_s / (d rho_s)
//   dh_s  = a_s dr + alpha_s w - beta_s h_s
//   dw   += sum_s alpha_s h_s                       (over all tokens)
//
// agg_bwd_ring_kernel (S <= 9, 16-byte aligned rows of at most 2 x 448
// vectors): the TMA ring of the forward kernels.  A token's rows arrive as
// [dr, h_0 .. h_{S-1}]; dr is copied to registers and its slot released at
// once, the source slots stay held between pass 1 (three partial sums per
// source, one warp reduce-scatter of 27 values, one cross-warp step) and
// pass 2 (dh_s written, this thread's share of dw accumulated in registers).
// Bytes per token: (S + 1) rows read, S rows written (plus S read with
// accumulate).
//
// agg_bwd_generic_kernel (everything else): one CTA per token at a time,
// plain loads, two passes.
//
// dw is deterministic: every CTA writes its partial sums to its own row of a
// caller-provided fp32 workspace [grid, d]; dw_reduce_kernel then adds the
// rows in a fixed order.
#include <atomic>
#include <math.h>

#include <mutex>

#include "ring_common.cuh"

namespace attnres {

constexpr int kBwdSmax = kRingSmax;
constexpr int kBwdVals = 3 * kBwdSmax;  // (w.h, h.h, dr.h) per source

struct BwdShared {
  uint64_t full[kRingMaxSlots];
  uint64_t empty[kRingMaxSlots];
  float red[2][kRingConsumerWarps][kBwdVals];
  int abort_flag[2];
};
constexpr int kBwdHeaderBytes = (int)((sizeof(BwdShared) + 127) / 128 * 128);

struct BwdParams {
  unsigned long long wait_ns;  // limit of each main-loop wait (the final drain keeps the default)
  int withhold_row1;           // bounded-wait test (as RingParams::withhold_row1)
  const char* src[kMaxSources];
  char* grad_src[kMaxSources];
  const char* grad_r;
  const float* w;
  float* ws;  // [gridDim.x, d]
  int* dev_err;
  long long T;
  int d;
  int S;
  int nvec;
  int row_bytes;
  int nslots;
  float eps;
  float inv_d;
};

// Producer of the backward ring: rows [dr, h_0 .. h_{S-1}] of each token.
// Rows per token, in ring order: grad_r, the S sources and, when the
// gradients accumulate, the S old gradient rows (read back through the ring
// like the rest, so pass 2 never waits on a plain load).  Pass 2 holds the
// source slots while it takes the old gradients: with nslots >= S + 1 the
// first old-gradient row always finds a free slot, and each later one a
// slot released by an earlier step of pass 2 (slots are reused in order).
template <bool ACC>
__device__ __forceinline__ void bwd_produce(const BwdParams& p, BwdShared& sh, uint32_t ring) {
  const int nslots = p.nslots;
  const int rows = ACC ? 2 * p.S + 1 : p.S + 1;
  uint32_t slot = 0, lap = 0;
  long long issued = 0;
  bool ok = true;
  for (long long t = blockIdx.x; t < p.T && ok; t += gridDim.x) {
    const long long off = t * (long long)p.row_bytes;
    for (int j = 0; j < rows; ++j) {
      const char* g = (j == 0 ? p.grad_r : j <= p.S ? p.src[j - 1] : p.grad_src[j - 1 - p.S]) + off;
      if (!mbar_wait_bounded(smem_addr(&sh.empty[slot]), (lap & 1u) ^ 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      const uint32_t full = smem_addr(&sh.full[slot]);
      mbar_arrive_expect_tx(full, (uint32_t)p.row_bytes);
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

template <typename T, int VPT, bool ACC>
__global__ void __launch_bounds__(kRingThreads, 1) agg_bwd_ring_kernel(const __grid_constant__ BwdParams p) {
  constexpr int EPV = Vec<T>::kElems;
  constexpr int NP = EPV / 2;
  extern __shared__ __align__(128) unsigned char smem[];
  BwdShared& sh = *reinterpret_cast<BwdShared*>(smem);
  const uint32_t ring = smem_addr(smem) + kBwdHeaderBytes;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nslots = p.nslots;
  if (tid == 0) {
    for (int k = 0; k < nslots; ++k) {
      mbar_init(smem_addr(&sh.full[k]), 1);
      mbar_init(smem_addr(&sh.empty[k]), kRingConsumerWarps);
    }
    sh.abort_flag[0] = 0;
    sh.abort_flag[1] = 0;
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();  // everything below may read what the previous kernel wrote
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done

  if (warp == kRingConsumerWarps) {
    if (lane == 0) bwd_produce<ACC>(p, sh, ring);
    return;
  }

  // ------------------------------------------------------------ consumers --
  uint64_t wp[VPT][NP], dwacc[VPT][NP];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * kRingConsumers;
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const bool in = v < p.nvec;
      wp[k][j] = f2_pack(in ? __ldg(p.w + v * EPV + 2 * j) : 0.f, in ? __ldg(p.w + v * EPV + 2 * j + 1) : 0.f);
      dwacc[k][j] = 0;
    }
  }
  const int my_idx = rs_lane_index<kBwdVals>(lane);
  const int S = p.S;
  uint32_t slot = 0, lap = 0;
  bool ok = true;
  auto wait_slot = [&](uint32_t sl, uint32_t parity) {
    if (ok && !mbar_wait_bounded(smem_addr(&sh.full[sl]), parity, p.wait_ns)) ok = false;
  };
  auto release = [&](uint32_t sl) {
    // Lane 0 releases the slot only while its own waits have all succeeded:
    // then this phase completed and its copy landed.  After a wait ran out
    // the copy may still be in flight, and the slot must not be refilled
    // under it (the producer then runs out of slots, stops and drains).
    __syncwarp();
    if (lane == 0 && ok) mbar_arrive(smem_addr(&sh.empty[sl]));
  };
  auto load_row = [&](uint32_t sl, uint4* dst) {
    const uint32_t base = ring + sl * (uint32_t)p.row_bytes;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * kRingConsumers;
      dst[k] = v < p.nvec ? ld_shared_v4(base + (uint32_t)v * 16u) : make_uint4(0, 0, 0, 0);
    }
  };

  int iter = 0;
  for (long long t = blockIdx.x; t < p.T; t += gridDim.x, ++iter) {
    const int buf = iter & 1;
    volatile int* abort_flag = &sh.abort_flag[buf];

    // the token's gradient row, kept in registers as fp32 pairs
    uint64_t drp[VPT][NP];
    {
      uint4 dv[VPT];
      wait_slot(slot, lap & 1u);
      load_row(slot, dv);
      release(slot);
      if (++slot == (uint32_t)nslots) { slot = 0; ++lap; }
#pragma unroll
      for (int k = 0; k < VPT; ++k) Vec<T>::pairs(dv[k], drp[k]);
    }

    // pass 1: w.h, h.h and dr.h of every source (slots stay held)
    const uint32_t first = slot;
    const uint32_t first_lap = lap;
    float part[kBwdVals];
#pragma unroll
    for (int s = 0; s < kBwdSmax; ++s) {
      part[3 * s] = 0.f;
      part[3 * s + 1] = 0.f;
      part[3 * s + 2] = 0.f;
      if (s < S) {
        uint4 hv[VPT];
        wait_slot(slot, lap & 1u);
        load_row(slot, hv);
        if (++slot == (uint32_t)nslots) { slot = 0; ++lap; }
        uint64_t q2 = 0, ss2 = 0, g2 = 0;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          uint64_t h[NP];
          Vec<T>::pairs(hv[k], h);
#pragma unroll
          for (int j = 0; j < NP; ++j) {
            q2 = f2_fma(wp[k][j], h[j], q2);
            ss2 = f2_fma(h[j], h[j], ss2);
            g2 = f2_fma(drp[k][j], h[j], g2);
          }
        }
        part[3 * s] = f2_hsum(q2);
        part[3 * s + 1] = f2_hsum(ss2);
        part[3 * s + 2] = f2_hsum(g2);
      }
    }
    (void)first_lap;

    reduce_scatter<kBwdVals>(part, lane);
    if (my_idx >= 0 && my_idx < 3 * S) sh.red[buf][warp][my_idx] = part[0];
    const bool warp_failed = __any_sync(0xffffffffu, !ok);
    if (lane == 0 && warp_failed) *abort_flag = 1;
    named_barrier_sync(kRingBarrierId, kRingConsumers);

    // coefficients (lane 3s holds source s; every warp computes them alike)
    const bool abort = *abort_flag != 0;
    float tot = 0.f;
    if (lane < 3 * S) {
#pragma unroll
      for (int w = 0; w < kRingConsumerWarps; ++w) tot += sh.red[buf][w][lane];
    }
    const float ssv = __shfl_down_sync(0xffffffffu, tot, 1);
    const float gv = __shfl_down_sync(0xffffffffu, tot, 2);
    const bool is_src = lane < 3 * S && lane % 3 == 0;
    // fast reciprocal square root, exponential and division: a few fp32 ulps
    const float inv_rho = rsqrtf(fmaf(ssv, p.inv_d, p.eps));
    const float z = is_src ? tot * inv_rho : -INFINITY;
    const float m = warp_max(z);
    const float e = is_src ? __expf(z - m) : 0.f;
    const float a = __fdividef(e, warp_sum(e));
    const float gbar = warp_sum(is_src ? a * gv : 0.f);
    const float nan = __int_as_float(0x7fc00000);
    const float dz = a * (gv - gbar);
    const float alpha = abort ? nan : dz * inv_rho;
    const float beta = abort ? nan : alpha * z * inv_rho * p.inv_d;
    const float aa = abort ? nan : a;

    // pass 2: dh_s = a_s dr + alpha_s w - beta_s h_s, dw += alpha_s h_s
    uint32_t sl = first;
#pragma unroll
    for (int s = 0; s < kBwdSmax; ++s) {
      if (s < S) {
        const float as = __shfl_sync(0xffffffffu, aa, 3 * s);
        const float al = __shfl_sync(0xffffffffu, alpha, 3 * s);
        const float be = __shfl_sync(0xffffffffu, beta, 3 * s);
        const uint64_t a2 = f2_pack(as, as), al2 = f2_pack(al, al), nbe2 = f2_pack(-be, -be);
        uint4 hv[VPT], gv[VPT];
        load_row(sl, hv);
        if (ACC) {
          // the old gradient row of source s, next in the ring
          wait_slot(slot, lap & 1u);
          load_row(slot, gv);
        }
        char* grow = p.grad_src[s] + t * (long long)p.row_bytes;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          const int v = tid + k * kRingConsumers;
          if (v < p.nvec) {
            uint64_t h[NP];
            Vec<T>::pairs(hv[k], h);
            float out[EPV];
            uint64_t old[NP];
            if (ACC) Vec<T>::pairs(gv[k], old);
#pragma unroll
            for (int j = 0; j < NP; ++j) {
              uint64_t dh = f2_fma(a2, drp[k][j], ACC ? old[j] : 0);
              dh = f2_fma(al2, wp[k][j], dh);
              dh = f2_fma(nbe2, h[j], dh);
              dwacc[k][j] = f2_fma(al2, h[j], dwacc[k][j]);
              f2_unpack(dh, out[2 * j], out[2 * j + 1]);
            }
            *reinterpret_cast<uint4*>(grow + (size_t)v * 16) = Vec<T>::pack(out);
          }
        }
        release(sl);
        if (++sl == (uint32_t)nslots) sl = 0;
        if (ACC) {
          release(slot);
          if (++slot == (uint32_t)nslots) { slot = 0; ++lap; }
        }
      }
    }
    if (abort) {
      if (tid == 0) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
      break;
    }
  }

  // this CTA's partial dw for its channels
  float* wrow = p.ws + (size_t)blockIdx.x * p.d;
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * kRingConsumers;
    if (v < p.nvec) {
#pragma unroll
      for (int j = 0; j < NP; ++j) {
        float lo, hi;
        f2_unpack(dwacc[k][j], lo, hi);
        wrow[v * EPV + 2 * j] = lo;
        wrow[v * EPV + 2 * j + 1] = hi;
      }
    }
  }
}

// ------------------------------------------------------------ generic ----

constexpr int kBwdGenThreads = 256;

template <typename T, bool ACC>
__global__ void __launch_bounds__(kBwdGenThreads) agg_bwd_generic_kernel(const __grid_constant__ BwdParams p) {
  __shared__ float s_red[kBwdGenThreads / 32][3];
  __shared__ float s_q[kMaxSources], s_ss[kMaxSources], s_g[kMaxSources];
  __shared__ float s_a[kMaxSources], s_al[kMaxSources], s_be[kMaxSources];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d = p.d, S = p.S;
  pdl_wait();
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done
  float* wrow = p.ws + (size_t)blockIdx.x * d;
  for (int c = tid; c < d; c += kBwdGenThreads) wrow[c] = 0.f;
  for (long long t = blockIdx.x; t < p.T; t += gridDim.x) {
    const long long row = t * (long long)d;
    const T* dr = reinterpret_cast<const T*>(p.grad_r) + row;
    for (int s = 0; s < S; ++s) {
      const T* h = reinterpret_cast<const T*>(p.src[s]) + row;
      float q = 0.f, ss = 0.f, g = 0.f;
      for (int c = tid; c < d; c += kBwdGenThreads) {
        const float x = load_elem(h + c);
        q = fmaf(p.w[c], x, q);
        ss = fmaf(x, x, ss);
        g = fmaf(load_elem(dr + c), x, g);
      }
      q = warp_sum(q);
      ss = warp_sum(ss);
      g = warp_sum(g);
      if (lane == 0) {
        s_red[warp][0] = q;
        s_red[warp][1] = ss;
        s_red[warp][2] = g;
      }
      __syncthreads();
      if (tid == 0) {
        float a0 = 0.f, a1 = 0.f, a2 = 0.f;
        for (int w = 0; w < kBwdGenThreads / 32; ++w) {
          a0 += s_red[w][0];
          a1 += s_red[w][1];
          a2 += s_red[w][2];
        }
        s_q[s] = a0;
        s_ss[s] = a1;
        s_g[s] = a2;
      }
      __syncthreads();
    }
    if (warp == 0) {
      float m = -INFINITY;
      for (int s = lane; s < S; s += 32) m = fmaxf(m, s_q[s] / sqrtf(s_ss[s] / (float)d + p.eps));
      m = warp_max(m);
      float tot = 0.f;
      for (int s = lane; s < S; s += 32) tot += expf(s_q[s] / sqrtf(s_ss[s] / (float)d + p.eps) - m);
      tot = warp_sum(tot);
      float gb = 0.f;
      for (int s = lane; s < S; s += 32) {
        const float rho = sqrtf(s_ss[s] / (float)d + p.eps);
        const float z = s_q[s] / rho;
        const float a = expf(z - m) / tot;
        s_a[s] = a;
        gb += a * s_g[s];
      }
      gb = warp_sum(gb);
      for (int s = lane; s < S; s += 32) {
        const float rho = sqrtf(s_ss[s] / (float)d + p.eps);
        const float z = s_q[s] / rho;
        const float al = s_a[s] * (s_g[s] - gb) / rho;
        s_al[s] = al;
        s_be[s] = al * z / (rho * (float)d);
      }
    }
    __syncthreads();
    for (int c = tid; c < d; c += kBwdGenThreads) {
      const float drc = load_elem(dr + c);
      const float wc = p.w[c];
      float dwc = 0.f;
      for (int s = 0; s < S; ++s) {
        const float x = load_elem(reinterpret_cast<const T*>(p.src[s]) + row + c);
        T* gp = reinterpret_cast<T*>(p.grad_src[s]) + row + c;
        float dh = s_a[s] * drc + s_al[s] * wc - s_be[s] * x;
        if (ACC) dh += load_elem(gp);
        store_elem(gp, dh);
        dwc = fmaf(s_al[s], x, dwc);
      }
      wrow[c] += dwc;
    }
    __syncthreads();
  }
}

// dw[c] = sum over the nb workspace rows of ws[b, c], in a fixed order: the
// kDwSplit threads of channel c each add rows b = part, part + kDwSplit, ...
// in turn (all their loads independent, so in flight together), then the
// kDwSplit partials are added in part order through shared memory.  A block
// covers 32 consecutive channels (coalesced 128-byte row segments).
constexpr int kDwSplit = 8;
constexpr int kDwThreads = 32 * kDwSplit;

__global__ void __launch_bounds__(kDwThreads) dw_reduce_kernel(const float* ws, int nb, int d, float* dw) {
  __shared__ float part_sum[kDwSplit][32];
  pdl_wait();
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done
  const int cl = threadIdx.x & 31;
  const int part = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + cl;
  float s = 0.f;
  if (c < d) {
#pragma unroll 8
    for (int b = part; b < nb; b += kDwSplit) s += ws[(size_t)b * d + c];
  }
  part_sum[part][cl] = s;
  __syncthreads();
  if (part == 0 && c < d) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < kDwSplit; ++k) t += part_sum[k][cl];
    dw[c] = t;
  }
}

// ---------------------------------------------------------------- launch --

template <typename T, int VPT, bool ACC>
static cudaError_t launch_bwd_ring_t(const BwdParams& bp, int grid, int smem, cudaStream_t stream) {
  static SmemOptIn optin;  // the large shared-memory opt-in, per device and context
  auto kern = agg_bwd_ring_kernel<T, VPT, ACC>;
  cudaError_t e = optin.ensure(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  e = launch_kernel(kern, dim3(grid), dim3(kRingThreads), (size_t)smem, stream, bp);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <typename T>
static cudaError_t launch_bwd_ring_vpt(const BwdParams& bp, int vpt, bool acc, int grid, int smem,
                                       cudaStream_t stream) {
  if (vpt == 1) {
    return acc ? launch_bwd_ring_t<T, 1, true>(bp, grid, smem, stream)
               : launch_bwd_ring_t<T, 1, false>(bp, grid, smem, stream);
  }
  return acc ? launch_bwd_ring_t<T, 2, true>(bp, grid, smem, stream)
             : launch_bwd_ring_t<T, 2, false>(bp, grid, smem, stream);
}

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t backward_blocks(int64_t T) {
  DeviceInfo di;
  if (device_info(&di) != cudaSuccess) return -1;
  return T < di.sm_count ? T : di.sm_count;
}

cudaError_t launch_aggregate_backward(const BwdArgs& a) {
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  const int grid = (int)backward_blocks(a.T);
  if (a.T <= 0 || grid <= 0) return cudaMemsetAsync(a.grad_w, 0, sizeof(float) * (size_t)a.d, a.stream);
  const bool bf16 = a.dtype == ATTNRES_BF16;
  const int esz = bf16 ? 2 : 4;
  const long long row_bytes = (long long)a.d * esz;

  BwdParams bp{};
  for (int s = 0; s < a.S; ++s) {
    bp.src[s] = static_cast<const char*>(a.src[s]);
    bp.grad_src[s] = static_cast<char*>(a.grad_src[s]);
  }
  bp.grad_r = static_cast<const char*>(a.grad_r);
  bp.w = a.w;
  bp.ws = a.workspace;
  bp.dev_err = a.dev_err;
  bp.T = a.T;
  bp.d = a.d;
  bp.S = a.S;
  bp.eps = a.eps;
  bp.inv_d = 1.0f / (float)a.d;
  bp.wait_ns = wait_limit_ns();
  bp.withhold_row1 = debug_withhold_row1();
  bp.row_bytes = (int)row_bytes;

  bool ring = a.S <= kBwdSmax && row_bytes % 16 == 0 && al16(a.grad_r);
  const long long nvec = row_bytes / 16;
  const int vpt = (int)((nvec + kRingConsumers - 1) / kRingConsumers);
  ring = ring && vpt >= 1 && vpt <= kRingMaxVpt;
  for (int s = 0; ring && s < a.S; ++s) ring = al16(a.src[s]) && al16(a.grad_src[s]);
  int nslots = 0;
  if (ring) {
    nslots = (int)(((long long)di.max_smem_optin - kBwdHeaderBytes) / row_bytes);
    if (nslots > kRingMaxSlots) nslots = kRingMaxSlots;
    ring = nslots >= a.S + 1;  // a token's rows must fit in the ring
  }
  if (ring) {
    bp.nvec = (int)nvec;
    bp.nslots = nslots;
    const int smem = kBwdHeaderBytes + nslots * (int)row_bytes;
    e = bf16 ? launch_bwd_ring_vpt<bf16_t>(bp, vpt, a.accumulate, grid, smem, a.stream)
             : launch_bwd_ring_vpt<float>(bp, vpt, a.accumulate, grid, smem, a.stream);
  } else {
    if (bf16) {
      e = a.accumulate ? launch_kernel(agg_bwd_generic_kernel<bf16_t, true>, dim3(grid), dim3(kBwdGenThreads), 0,
                                       a.stream, bp)
                       : launch_kernel(agg_bwd_generic_kernel<bf16_t, false>, dim3(grid), dim3(kBwdGenThreads), 0,
                                       a.stream, bp);
    } else {
      e = a.accumulate ? launch_kernel(agg_bwd_generic_kernel<float, true>, dim3(grid), dim3(kBwdGenThreads), 0,
                                       a.stream, bp)
                       : launch_kernel(agg_bwd_generic_kernel<float, false>, dim3(grid), dim3(kBwdGenThreads), 0,
                                       a.stream, bp);
    }
  }
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rgrid = (a.d + 31) / 32;
  e = launch_kernel(dw_reduce_kernel, dim3(rgrid), dim3(kDwThreads), 0, a.stream, (const float*)a.workspace, grid, a.d,
                    a.grad_w);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ------------------------------------------- backward without allocation --
//
// For callers that cannot allocate device memory (for instance code running
// inside a graph-replay or real-time serving loop with a fixed memory budget,
// or a host that forbids cudaMalloc after start-up): the backward's fp32
// workspace lives in this file-scope array instead of a caller buffer.  It is
// part of the library's module, so every GPU that loads the library holds it
// until the process exits.  Every call shares it and it keeps the previous
// call's contents; the backward writes every element it later reads, so
// nothing has to be cleared.  Calls whose kernels overlap on a GPU race on it.
constexpr int64_t kNoAllocScratchFloats = 160 * 8192;  // 5 MiB: 160 CTA rows of d <= 8192
static __device__ __align__(256) float g_noalloc_bwd_scratch[kNoAllocScratchFloats];

// Device address of the scratch array on the current device (a host-side
// name of a __device__ array is not a device address).  Looked up with
// cudaGetSymbolAddress the first time on a device, and again whenever the
// device's context has changed since (a reset reloads the module at a new
// address); otherwise the cached address is used.
cudaError_t noalloc_backward_scratch(float** ptr, int64_t* capacity_floats) {
  constexpr int kMaxDevices = 64;
  static float* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  static std::mutex lock;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> guard(lock);
  if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_bwd_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<float*>(p);
    ctx_of[dev] = current_context_id();  // the lookup made the device's context current on this thread
  }
  *ptr = addr[dev];
  *capacity_floats = kNoAllocScratchFloats;
  return cudaSuccess;
}

}  // namespace attnres
