// Two-phase schedule of Block AttnRes inference (Kimi K3 chaptered tutorial,
// ch. 4.4 and 4.6): the cached block sums [h_0, b_1 .. b_{n-1}] are fixed for
// the whole of block n, so one batched inter-block pass reads each of them
// once and aggregates them for every layer query of the block; each layer
// then folds in its own partial sum with an online-softmax merge.
//
//  agg_interblock_kernel (phase 1): the TMA ring of the aggregation kernels
//      (ring_common.cuh) brings a token's n <= 9 cached rows into shared
//      memory, where they stay until the token is done.  Phase A: the
//      Q x n logits and the n sums of squares, queries taken two at a time
//      (each row vector is unpacked once per pair of queries), each pair's
//      per-thread partials summed over the warp by one reduce-scatter and
//      over the warps in shared memory.  One barrier, then the softmax of
//      every query (one warp per query), one more barrier, then phase C:
//      the Q weighted sums, four queries at a time (each row vector
//      unpacked once per four queries), written as fp32 rows.
//
//  agg_merge_kernel (phase 2, one layer): p = round(prev + F) (or F) is
//      stored as the new partial sum / block sum, its logit z_p = w.p/rms(p)
//      is reduced over the CTA, and with m = max(lse, z_p)
//          r = (e^{lse - m} r_inter + e^{z_p - m} p) / (e^{lse - m} + e^{z_p - m})
//      weights: the inter-block ones scaled by e^{lse - m}/den, e^{z_p - m}/den
//      for the partial.  Without a partial (first layer of a block) r is
//      r_inter itself.
#include <atomic>
#include <math.h>

#include "ring_common.cuh"

namespace attnres {

// Bring the cache line holding p into L1 ahead of its use (no register
// holds the data; a later load of the line then hits).
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

struct InterParams {
  RingParams rp;  // the cached sources (n_stored = S = n), geometry, ring
  const float* wq[kMaxQueries];
  int Q;
  float* out_r;    // [Q, T, d] fp32
  float* out_lse;  // [Q, T]
  float* out_a;    // [Q, T, n] or null
  char* out_r0;    // [T, d] of the sources' type or null: query 0's row, rounded (a block's first layer)
  float* out_a0;   // [T, n] or null: query 0's weights
  const float* dots;  // DOTS kernels: partial dot products w_q . h_s, [ksplit][T][n][Q]
  int ksplit;
  int tail_groups;  // DOTS kernels: query groups each of the last T mod grid tokens is split into
};

// The DOTS kernels' work units.  CTA b first takes whole tokens b, b + G,
// ... (G = gridDim.x) while a full round of G tokens remains; the r < G
// tokens left over are split into g = tail_groups query groups each, so
// that r g <= G CTAs share the last round: CTA b < r g takes token
// T_full + b / g, queries [(b mod g) Q / g, (b mod g + 1) Q / g).  Unit k of
// this CTA: false once there is none.
__device__ __forceinline__ bool inter_unit(const InterParams& ip, int k, long long* t, int* qlo, int* qhi) {
  const long long G = gridDim.x, b = blockIdx.x;
  const long long rounds = ip.rp.T / G;
  if (k < rounds) {
    *t = b + k * G;
    *qlo = 0;
    *qhi = ip.Q;
    return true;
  }
  const long long r = ip.rp.T - rounds * G;
  const int g = ip.tail_groups;
  if (k > rounds || b >= r * g) return false;
  const int grp = (int)(b % g);
  *t = rounds * G + b / g;
  *qlo = grp * ip.Q / g;
  *qhi = (grp + 1) * ip.Q / g;
  return true;
}

// The producer of the DOTS kernels: every source row of this CTA's units'
// tokens, in unit order (otherwise as ring_produce).  The kernel before a
// DOTS kernel is always the tensor-core logits kernel, which waits for its
// own predecessor before it lets this one launch: the sources, written
// before that, are complete when this kernel starts.  So the rows fill the
// ring before the wait for the logits kernel, which comes only when the
// ring is full (and precedes the signal to this kernel's dependents).
__device__ __forceinline__ void inter_produce(const InterParams& ip, RingShared& sh, uint32_t ring) {
  const RingParams& p = ip.rp;
  const int nslots = p.nslots;
  uint32_t slot = 0, lap = 0;
  long long issued = 0;
  bool ok = true, waited = false;
  long long t;
  int qlo, qhi;
  for (int k = 0; ok && inter_unit(ip, k, &t, &qlo, &qhi); ++k) {
    const long long off = t * (long long)p.row_bytes;
    for (int j = 0; j < p.S; ++j) {
      if (!waited && issued == nslots) {
        pdl_wait();
        pdl_trigger();
        waited = true;
      }
      if (!mbar_wait_bounded(smem_addr(&sh.empty[slot]), (lap & 1u) ^ 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      const uint32_t full = smem_addr(&sh.full[slot]);
      mbar_arrive_expect_tx(full, (uint32_t)p.row_bytes);
      // the bounded-wait test arms one row of the first token without its copy
      if (issued + 1 != p.withhold_row1)
        bulk_copy_g2s(ring + slot * (uint32_t)p.row_bytes, p.src[j] + off, (uint32_t)p.row_bytes, full);
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

// 4 bytes global -> shared without a register (cp.async, cached in L1);
// complete after cp_async_commit and cp_async_wait_all in the same thread.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// A block's first layer takes query 0's row as its output: the merge
// computes it as 1 * r + 0 before rounding (which turns a -0 into +0);
// these give the same bits when the pass writes that output itself.
__device__ __forceinline__ float first_layer_value(float r) { return fmaf(1.0f, r, 0.0f); }

constexpr int kInterGA = 2;  // queries per phase-A group (the logits)
constexpr int kInterMaxSplit = 16;  // channel splits of the tensor-core logits, at most
constexpr int kInterGC = 4;  // queries per phase-C group (the weighted sums)
constexpr int kInterSumsq = kMaxQueries * kRingSmax;  // offset of the sums of squares in a warp's partials

// Shared memory between the ring header and the ring slots.
constexpr int kInterA2Row = kRingSmax + 1;  // 10 pairs: 80-byte rows, 16-byte aligned
struct InterShared {
  float2 a2[kMaxQueries][kInterA2Row];  // softmax weights as (a, a) pairs
  union {
    float red[kRingConsumerWarps][kInterSumsq + kRingSmax];  // per-warp totals: logits [q * 9 + s], then sums of squares
    // with precomputed dots: the token's partial dots [q][split][s], each
    // element copied in (cp.async) and summed by the thread that needs it
    float pd[kMaxQueries][kInterMaxSplit][kRingSmax];
  };
  float ss[kRingConsumerWarps][kRingSmax];  // per-warp sums of squares (precomputed-dots kernel)
};
constexpr int kInterSharedBytes = (int)((sizeof(InterShared) + 127) / 128 * 128);

template <typename Tin, int VPT, bool EXACT>
__global__ void __launch_bounds__(kRingThreads, 1) agg_interblock_kernel(const __grid_constant__ InterParams ip) {
  const RingParams& p = ip.rp;
  constexpr int EPV = Vec<Tin>::kElems;
  constexpr int NP = EPV / 2;
  extern __shared__ __align__(128) unsigned char smem[];
  RingShared& sh = *reinterpret_cast<RingShared*>(smem);
  InterShared& xs = *reinterpret_cast<InterShared*>(smem + kRingHeaderBytes);
  const uint32_t ring = smem_addr(smem) + kRingHeaderBytes + kInterSharedBytes;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nslots = p.nslots;
  ring_init(p, sh);
  __syncthreads();
  pdl_wait();
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done

  if (warp == kRingConsumerWarps) {
    if (lane == 0) ring_produce(p, sh, ring);
    return;
  }

  const int S = p.S;
  const int Q = ip.Q;
  const long long T = p.T;
  const float nan = __int_as_float(0x7fc00000);
  uint32_t slot = 0, lap = 0;  // ring position of the next token's first row
  bool ok = true;
  int iter = 0;
  bool abort = false;
  for (long long t = blockIdx.x; t < T && !abort; t += gridDim.x, ++iter) {
    const int buf = iter & 1;
    volatile int* abort_flag = &sh.abort_flag[buf];
    // wait for the token's n rows; they stay in their slots until phase C
    // is done with them
    uint32_t row[kRingSmax];  // shared-memory address of source s's row
    uint32_t sl_of[kRingSmax];
#pragma unroll
    for (int s = 0; s < kRingSmax; ++s) {
      row[s] = 0;
      sl_of[s] = 0;
      if (s < S) {
        uint32_t sl = slot + s, lp = lap;
        if (sl >= (uint32_t)nslots) {
          sl -= nslots;
          ++lp;
        }
        if (ok && !mbar_wait_bounded(smem_addr(&sh.full[sl]), lp & 1u, p.wait_ns)) ok = false;
        row[s] = ring + sl * (uint32_t)p.row_bytes;
        sl_of[s] = sl;
      }
    }

    // ---- phase A: logits of every query and the sums of squares
    for (int q0 = 0; q0 < Q; q0 += kInterGA) {
      const bool first = q0 == 0;
      uint64_t acc[kInterGA][kRingSmax];
      uint64_t ss2[kRingSmax];
#pragma unroll
      for (int s = 0; s < kRingSmax; ++s) {
        ss2[s] = 0;
#pragma unroll
        for (int g = 0; g < kInterGA; ++g) acc[g][s] = 0;
      }
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = tid + k * kRingConsumers;
        if (EXACT || v < p.nvec) {
          uint64_t wp[kInterGA][NP];
#pragma unroll
          for (int g = 0; g < kInterGA; ++g) {
            const bool qin = q0 + g < Q;
#pragma unroll
            for (int j = 0; j < NP; j += 2) {
              const float4 w4 = qin ? __ldg(reinterpret_cast<const float4*>(ip.wq[q0 + g] + v * EPV + 2 * j))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
              wp[g][j] = f2_pack(w4.x, w4.y);
              wp[g][j + 1] = f2_pack(w4.z, w4.w);
            }
          }
#pragma unroll
          for (int s = 0; s < kRingSmax; ++s) {
            if (s < S) {
              uint64_t h[NP];
              Vec<Tin>::pairs(ld_shared_v4(row[s] + (uint32_t)v * 16u), h);
#pragma unroll
              for (int j = 0; j < NP; ++j) {
#pragma unroll
                for (int g = 0; g < kInterGA; ++g) acc[g][s] = f2_fma(wp[g][j], h[j], acc[g][s]);
                if (first) ss2[s] = f2_fma(h[j], h[j], ss2[s]);
              }
            }
          }
        }
      }
      // this warp's totals: one reduce-scatter of the pair's 2 x 9 logits
      // (and, for the first pair, the 9 sums of squares)
      float part[kInterGA * kRingSmax + kRingSmax];
#pragma unroll
      for (int g = 0; g < kInterGA; ++g)
#pragma unroll
        for (int s = 0; s < kRingSmax; ++s) part[g * kRingSmax + s] = f2_hsum(acc[g][s]);
      if (first) {
        constexpr int N = kInterGA * kRingSmax + kRingSmax;
#pragma unroll
        for (int s = 0; s < kRingSmax; ++s) part[kInterGA * kRingSmax + s] = f2_hsum(ss2[s]);
        reduce_scatter<N>(part, lane);
        const int idx = rs_lane_index<N>(lane);
        if (idx >= 0) {
          const int g = idx / kRingSmax, s = idx % kRingSmax;
          if (g < kInterGA) {
            if (s < S && q0 + g < Q) xs.red[warp][(q0 + g) * kRingSmax + s] = part[0];
          } else if (s < S) {
            xs.red[warp][kInterSumsq + s] = part[0];
          }
        }
      } else {
        constexpr int N = kInterGA * kRingSmax;
        reduce_scatter<N>(part, lane);
        const int idx = rs_lane_index<N>(lane);
        if (idx >= 0) {
          const int g = idx / kRingSmax, s = idx % kRingSmax;
          if (s < S && q0 + g < Q) xs.red[warp][(q0 + g) * kRingSmax + s] = part[0];
        }
      }
    }
    const bool warp_failed = __any_sync(0xffffffffu, !ok);
    if (lane == 0 && warp_failed) *abort_flag = 1;
    named_barrier_sync(kRingBarrierId, kRingConsumers);

    // the CTA-uniform exit test: every warp reads the flag after the barrier
    abort = *abort_flag != 0;
    if (abort) {
      // the token is abandoned: NaN for every output of it, and no slot is
      // released (a copy may still be landing in one)
      float r[EPV];
#pragma unroll
      for (int e = 0; e < EPV; ++e) r[e] = nan;
      if (ip.out_r0) {
        char* r0row = ip.out_r0 + t * (long long)p.d * (long long)sizeof(Tin);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          const int v = tid + k * kRingConsumers;
          if (EXACT || v < p.nvec) store_out<Tin, EPV>(r0row, v, r);
        }
      }
      for (int q = 0; q < Q; ++q) {
        char* orow = reinterpret_cast<char*>(ip.out_r) + ((long long)q * T + t) * (long long)p.d * 4;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          const int v = tid + k * kRingConsumers;
          if (EXACT || v < p.nvec) store_out<float, EPV>(orow, v, r);
        }
      }
      if (warp == 0) {
        for (int q = lane; q < Q; q += 32) ip.out_lse[(long long)q * T + t] = nan;
        if (ip.out_a)
          for (int i = lane; i < Q * S; i += 32) ip.out_a[((long long)(i / S) * T + t) * S + i % S] = nan;
        if (ip.out_a0)
          for (int s2 = lane; s2 < S; s2 += 32) ip.out_a0[t * S + s2] = nan;
      }
      if (tid == 0) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
      break;
    }

    // ---- softmax of each query over the n sources (one warp per query)
    for (int q = warp; q < Q; q += kRingConsumerWarps) {
      const bool is_src = lane < S;
      float dot = 0.f, ss = 0.f;
      if (is_src) {
#pragma unroll
        for (int w = 0; w < kRingConsumerWarps; ++w) {
          dot += xs.red[w][q * kRingSmax + lane];
          ss += xs.red[w][kInterSumsq + lane];
        }
      }
      // fast reciprocal square root, exponential, logarithm and division:
      // a few fp32 ulps, far inside the parity tolerances
      const float z = is_src ? dot * rsqrtf(fmaf(ss, p.inv_d, p.eps)) : -INFINITY;
      const float m = warp_max(z);
      const float e = is_src ? __expf(z - m) : 0.f;
      const float esum = warp_sum(e);
      const float a = __fdividef(e, esum);
      if (is_src) {
        xs.a2[q][lane] = make_float2(a, a);
        if (ip.out_a) ip.out_a[((long long)q * T + t) * S + lane] = a;
        if (q == 0 && ip.out_a0) ip.out_a0[t * S + lane] = a;
      }
      if (lane == 0) ip.out_lse[(long long)q * T + t] = m + __logf(esum);
    }
    named_barrier_sync(kRingBarrierId, kRingConsumers);

    // ---- phase C: the weighted sums, four queries at a time
    for (int q0 = 0; q0 < Q; q0 += kInterGC) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = tid + k * kRingConsumers;
        if (EXACT || v < p.nvec) {
          uint64_t acc[kInterGC][NP];
#pragma unroll
          for (int g = 0; g < kInterGC; ++g)
#pragma unroll
            for (int j = 0; j < NP; ++j) acc[g][j] = 0;
#pragma unroll
          for (int s = 0; s < kRingSmax; ++s) {
            if (s < S) {
              uint64_t h[NP];
              Vec<Tin>::pairs(ld_shared_v4(row[s] + (uint32_t)v * 16u), h);
#pragma unroll
              for (int g = 0; g < kInterGC; ++g) {
                if (q0 + g < Q) {
                  const float2 ag = xs.a2[q0 + g][s];
                  const uint64_t a2 = f2_pack(ag.x, ag.y);
#pragma unroll
                  for (int j = 0; j < NP; ++j) acc[g][j] = f2_fma(a2, h[j], acc[g][j]);
                }
              }
            }
          }
#pragma unroll
          for (int g = 0; g < kInterGC; ++g) {
            if (q0 + g < Q) {
              float r[EPV];
#pragma unroll
              for (int j = 0; j < NP; ++j) f2_unpack(acc[g][j], r[2 * j], r[2 * j + 1]);
              char* orow = reinterpret_cast<char*>(ip.out_r) + ((long long)(q0 + g) * T + t) * (long long)p.d * 4;
              store_out<float, EPV>(orow, v, r);
              if (q0 + g == 0 && ip.out_r0) {
#pragma unroll
                for (int e = 0; e < EPV; ++e) r[e] = first_layer_value(r[e]);
                store_out<Tin, EPV>(ip.out_r0 + t * (long long)p.d * (long long)sizeof(Tin), v, r);
              }
            }
          }
        }
      }
    }

    // ---- release the token's slots.  Lane 0 releases a slot only while its
    // own waits have all succeeded: then the phase completed and its copy
    // landed.  After a wait ran out the copy may still be in flight, and the
    // slot must not be refilled under it (the producer then runs out of
    // slots, stops and drains).
    __syncwarp();
#pragma unroll
    for (int s = 0; s < kRingSmax; ++s) {
      if (s < S && lane == 0 && ok) mbar_arrive(smem_addr(&sh.empty[sl_of[s]]));
    }
    slot += S;
    if (slot >= (uint32_t)nslots) {
      slot -= nslots;
      ++lap;
    }
  }
}

// The inter-block pass when the dot products w_q . h_s come precomputed
// (the tensor-core kernel of twophase_tc.cu, partial sums per channel split
// in ip.dots, [ksplit][T][n][Q]); bf16 sources.  A consumer thread owns
// QPT quads of 4 channels (quad tid + m * 448), so that a warp's shared
// loads read 256 contiguous bytes and its fp32 stores write 512 contiguous
// bytes.  It takes its quads of the token's n rows into registers (the
// first KR sources; the others stay in their slots until the weighted sums
// are done) and releases the slots at once (the producer keeps the ring
// full), forming the sums of squares on the way.  At the token's start its
// warp's partial dots (queries warp, warp + 14) are copied into shared
// memory asynchronously, to be summed in split order in the softmax.  One
// barrier, the softmax of every query (one warp per query), one more
// barrier, then the weighted sums from registers: quad by quad, the n rows'
// 4 channels unpacked once, then every query's sum over them with its
// weights read two sources per shared load.  NS > 0 fixes the source count
// at compile time (no per-source branches in the inner loop).

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

template <int QPT, bool EXACT, int NS>
__global__ void __launch_bounds__(kRingThreads, 1) agg_interblock_dots_kernel(const __grid_constant__ InterParams ip) {
  const RingParams& p = ip.rp;
  extern __shared__ __align__(128) unsigned char smem[];
  RingShared& sh = *reinterpret_cast<RingShared*>(smem);
  InterShared& xs = *reinterpret_cast<InterShared*>(smem + kRingHeaderBytes);
  const uint32_t ring = smem_addr(smem) + kRingHeaderBytes + kInterSharedBytes;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nslots = p.nslots;
  const int nquad = 2 * p.nvec;  // 8-byte quads (4 bf16) per row
  ring_init(p, sh);
  __syncthreads();

  if (warp == kRingConsumerWarps) {
    // the producer streams the rows before it waits for the logits kernel
    if (lane == 0) inter_produce(ip, sh, ring);
    pdl_wait();
    pdl_trigger();
    return;
  }
  pdl_wait();  // the partial dots come from the logits kernel
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done

  const int S = NS > 0 ? NS : p.S;
  // sources whose quads stay in registers: the most that fit, with the n
  // unpacked sources of one quad, under the 128-register cap without spills
  // (5 up to n = 8, 4 at n = 9 or when n is known only at run time)
  constexpr int KR = NS == 0 ? (QPT > 2 ? 4 : kRingSmax) : (NS <= 5 ? NS : (NS == 9 ? 4 : 5));
  const int Q = ip.Q;
  const long long T = p.T;
  const float nan = __int_as_float(0x7fc00000);
  uint32_t slot = 0, lap = 0;
  bool ok = true;
  int iter = 0;
  bool abort = false;
  // Takes this thread's quads of the next ring slot into dst.  With
  // `release` the slot goes back to the producer at once; otherwise its
  // index is returned and the caller releases it after its last read.
  auto consume = [&](uint2* dst, bool release) -> uint32_t {
    if (ok && !mbar_wait_bounded(smem_addr(&sh.full[slot]), lap & 1u, p.wait_ns)) ok = false;
    const uint32_t taken = slot;
    const uint32_t base = ring + slot * (uint32_t)p.row_bytes;
#pragma unroll
    for (int m = 0; m < QPT; ++m) {
      const int qd = tid + m * kRingConsumers;
      dst[m] = (EXACT || qd < nquad) ? ld_shared_v2(base + (uint32_t)qd * 8u) : make_uint2(0, 0);
    }
    // Lane 0 releases the slot only while its own waits have all succeeded:
    // then this phase completed and its copy landed.  After a wait ran out
    // the copy may still be in flight, and the slot must not be refilled
    // under it (the producer then runs out of slots, stops and drains).
    if (release) {
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(smem_addr(&sh.empty[slot]));
    }
    if (++slot == (uint32_t)nslots) {
      slot = 0;
      ++lap;
    }
    return taken;
  };
  // the 4 channels of a quad as 2 packed fp32 pairs
  auto pairs = [](const uint2& v, uint64_t* h) {
    h[0] = f2_pack(bf16lo(v.x), bf16hi(v.x));
    h[1] = f2_pack(bf16lo(v.y), bf16hi(v.y));
  };

  long long t;
  int qlo, qhi;  // this unit's queries
  for (int unit = 0; !abort && inter_unit(ip, unit, &t, &qlo, &qhi); ++unit, ++iter) {
    const int buf = iter & 1;
    volatile int* abort_flag = &sh.abort_flag[buf];
    // this warp's queries' partial dots (queries warp, warp + 14; lane =
    // source), copied into shared memory without holding registers or
    // stalling: summed in the softmax, by the same thread
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int q = warp + u * kRingConsumerWarps;
      if (q >= qlo && q < qhi && lane < S) {
        for (int k = 0; k < ip.ksplit; ++k)
          cp_async_4(smem_addr(&xs.pd[q][k][lane]), ip.dots + (((long long)k * T + t) * S + lane) * Q + q);
      }
    }
    cp_async_commit();
    // the token's rows into registers (the first KR sources; the rest stay
    // in their slots until the weighted sums are done), the sums of squares
    // on the way
    uint2 x[KR][QPT];
    uint32_t held[kRingSmax];
    float part[kRingSmax];
#pragma unroll
    for (int s = 0; s < kRingSmax; ++s) {
      part[s] = 0.f;
      held[s] = 0;
      if (s < S) {
        uint2 xs_[QPT];
        if (s < KR)
          consume(x[s], true);
        else
          held[s] = consume(xs_, false);
        uint64_t ss2 = 0;
#pragma unroll
        for (int m = 0; m < QPT; ++m) {
          uint64_t h[2];
          pairs(s < KR ? x[s][m] : xs_[m], h);
          ss2 = f2_fma(h[0], h[0], ss2);
          ss2 = f2_fma(h[1], h[1], ss2);
        }
        part[s] = f2_hsum(ss2);
      }
    }
    reduce_scatter<kRingSmax>(part, lane);
    {
      const int idx = rs_lane_index<kRingSmax>(lane);
      if (idx >= 0 && idx < S) xs.ss[warp][idx] = part[0];
    }
    const bool warp_failed = __any_sync(0xffffffffu, !ok);
    if (lane == 0 && warp_failed) *abort_flag = 1;
    named_barrier_sync(kRingBarrierId, kRingConsumers);

    // the CTA-uniform exit test: every warp reads the flag after the barrier
    abort = *abort_flag != 0;
    if (abort) {
      for (int q = qlo; q < qhi; ++q) {
        char* orow = reinterpret_cast<char*>(ip.out_r) + ((long long)q * T + t) * (long long)p.d * 4;
#pragma unroll
        for (int m = 0; m < QPT; ++m) {
          const int qd = tid + m * kRingConsumers;
          if (EXACT || qd < nquad) *reinterpret_cast<float4*>(orow + (size_t)qd * 16) = make_float4(nan, nan, nan, nan);
        }
      }
      if (qlo == 0 && ip.out_r0) {
        char* r0row = ip.out_r0 + t * (long long)p.d * 2;
#pragma unroll
        for (int m = 0; m < QPT; ++m) {
          const int qd = tid + m * kRingConsumers;
          if (EXACT || qd < nquad) *reinterpret_cast<uint2*>(r0row + (size_t)qd * 8) = make_uint2(0x7fc07fc0u, 0x7fc07fc0u);
        }
      }
      if (warp == 0) {
        for (int q = qlo + lane; q < qhi; q += 32) ip.out_lse[(long long)q * T + t] = nan;
        if (ip.out_a)
          for (int i = qlo * S + lane; i < qhi * S; i += 32) ip.out_a[((long long)(i / S) * T + t) * S + i % S] = nan;
        if (qlo == 0 && ip.out_a0)
          for (int s2 = lane; s2 < S; s2 += 32) ip.out_a0[t * S + s2] = nan;
      }
      if (tid == 0) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
      cp_async_wait_all();  // no copy outlives the CTA
      break;
    }

    // ---- softmax of each query over the n sources (one warp per query)
    cp_async_wait_all();  // this thread's partial dots
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int q = warp + u * kRingConsumerWarps;
      if (q >= qlo && q < qhi) {
        const bool is_src = lane < S;
        float ss = 0.f, dot = 0.f;
        if (is_src) {
#pragma unroll
          for (int w = 0; w < kRingConsumerWarps; ++w) ss += xs.ss[w][lane];
          for (int k = 0; k < ip.ksplit; ++k) dot += xs.pd[q][k][lane];  // split order
        }
        // fast reciprocal square root, exponential, logarithm and division:
        // a few fp32 ulps, far inside the parity tolerances
        const float z = is_src ? dot * rsqrtf(fmaf(ss, p.inv_d, p.eps)) : -INFINITY;
        const float m = warp_max(z);
        const float e = is_src ? __expf(z - m) : 0.f;
        const float esum = warp_sum(e);
        const float a = __fdividef(e, esum);
        if (is_src) {
          xs.a2[q][lane] = make_float2(a, a);
          if (ip.out_a) ip.out_a[((long long)q * T + t) * S + lane] = a;
          if (q == 0 && ip.out_a0) ip.out_a0[t * S + lane] = a;
        }
        if (lane == 0) ip.out_lse[(long long)q * T + t] = m + __logf(esum);
      }
    }
    named_barrier_sync(kRingBarrierId, kRingConsumers);

    // ---- the weighted sums from registers, one quad at a time
    const long long qstride = T * (long long)p.d * 4;  // bytes between queries' rows
#pragma unroll
    for (int m = 0; m < QPT; ++m) {
      const int qd = tid + m * kRingConsumers;
      if (EXACT || qd < nquad) {
        uint64_t h[kRingSmax][2];
#pragma unroll
        for (int s = 0; s < kRingSmax; ++s) {
          if (s < S && s < KR) pairs(x[s][m], h[s]);
          if (s < S && s >= KR) pairs(ld_shared_v2(ring + held[s] * (uint32_t)p.row_bytes + (uint32_t)qd * 8u), h[s]);
        }
        char* orow = reinterpret_cast<char*>(ip.out_r) + (t * (long long)p.d + (long long)qd * 4) * 4;
#pragma unroll 4
        for (int q = qlo; q < qhi; ++q) {
          const float4* aq = reinterpret_cast<const float4*>(&xs.a2[q][0]);
          uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
          for (int s2 = 0; s2 < kInterA2Row / 2; ++s2) {
            if (2 * s2 < S) {
              const float4 w = aq[s2];  // (a_s, a_s, a_s+1, a_s+1)
              const uint64_t wa = f2_pack(w.x, w.y);
              acc0 = f2_fma(wa, h[2 * s2][0], acc0);
              acc1 = f2_fma(wa, h[2 * s2][1], acc1);
              if (2 * s2 + 1 < S) {
                const uint64_t wb = f2_pack(w.z, w.w);
                acc0 = f2_fma(wb, h[2 * s2 + 1][0], acc0);
                acc1 = f2_fma(wb, h[2 * s2 + 1][1], acc1);
              }
            }
          }
          float4 r;
          f2_unpack(acc0, r.x, r.y);
          f2_unpack(acc1, r.z, r.w);
          __stcs(reinterpret_cast<float4*>(orow + q * qstride), r);  // streamed: evict first from L2
          if (q == 0 && ip.out_r0)  // the block's first layer, in the sources' bf16
            *reinterpret_cast<uint2*>(ip.out_r0 + (t * (long long)p.d + (long long)qd * 4) * 2) =
                make_uint2(pack_bf16x2(first_layer_value(r.x), first_layer_value(r.y)),
                           pack_bf16x2(first_layer_value(r.z), first_layer_value(r.w)));
        }
      }
    }
    // the held slots back to the producer (same rule as in consume)
    __syncwarp();
#pragma unroll
    for (int s = KR; s < kRingSmax; ++s)
      if (s < S && lane == 0 && ok) mbar_arrive(smem_addr(&sh.empty[held[s]]));
  }
}

// ------------------------------------------------------------- phase 2 ---

constexpr int kMergeThreads = kRingConsumers;  // 448: two 16-byte vectors each at d = 7168 bf16

struct MergeParams {
  const char* prev;  // partial sum before this layer, or null
  const char* F;     // output of the previous layer, or null (first layer of a block)
  char* dst;         // new partial sum / block sum (when F)
  const float* w;
  const float* r_inter;  // [T, d]
  const float* lse_inter;  // [T]
  const float* a_inter;  // [T, n] or null
  char* out_r;
  float* out_a;  // [T, n + (F ? 1 : 0)] or null
  long long T;
  int d;
  int n;  // cached sources
  int nvec;
  float eps;
  float inv_d;
};

template <typename Tin, int VPT>
__global__ void __launch_bounds__(kMergeThreads) agg_merge_kernel(const __grid_constant__ MergeParams p) {
  constexpr int EPV = Vec<Tin>::kElems;
  constexpr int NP = EPV / 2;
  __shared__ float s_red[kMergeThreads / 32][2];
  __shared__ float s_c[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done
  const bool has_p = p.F != nullptr;
  uint64_t wp[VPT][NP];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int v = tid + k * kMergeThreads;
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const bool in = has_p && v < p.nvec;
      wp[k][j] = f2_pack(in ? __ldg(p.w + v * EPV + 2 * j) : 0.f, in ? __ldg(p.w + v * EPV + 2 * j + 1) : 0.f);
    }
  }
  const long long row_bytes = (long long)p.d * (long long)sizeof(Tin);
  for (long long t = blockIdx.x; t < p.T; t += gridDim.x) {
    // the inter-block row does not depend on this token's reduction: its
    // lines are prefetched into L1 first (no registers held), so one DRAM
    // round trip covers both inputs
    const float* rrow = p.r_inter + t * (long long)p.d;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * kMergeThreads;
      if (v < p.nvec) prefetch_l1(rrow + v * EPV);
    }
    uint4 x[VPT];
    float c1 = 1.f, c2 = 0.f;
    if (has_p) {
      uint64_t dot2 = 0, ss2 = 0;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int v = tid + k * kMergeThreads;
        x[k] = make_uint4(0, 0, 0, 0);
        if (v < p.nvec) {
          float f[EPV];
          Vec<Tin>::unpack(*reinterpret_cast<const uint4*>(p.F + t * row_bytes + (size_t)v * 16), f);
          if (p.prev) {
            float q[EPV];
            Vec<Tin>::unpack(*reinterpret_cast<const uint4*>(p.prev + t * row_bytes + (size_t)v * 16), q);
#pragma unroll
            for (int e = 0; e < EPV; ++e) f[e] = q[e] + f[e];
          }
          x[k] = Vec<Tin>::pack(f);  // one rounding to the storage type
          *reinterpret_cast<uint4*>(p.dst + t * row_bytes + (size_t)v * 16) = x[k];
          uint64_t h[NP];
          Vec<Tin>::pairs(x[k], h);
#pragma unroll
          for (int j = 0; j < NP; ++j) {
            dot2 = f2_fma(wp[k][j], h[j], dot2);
            ss2 = f2_fma(h[j], h[j], ss2);
          }
        }
      }
      float dot = warp_sum(f2_hsum(dot2));
      float ss = warp_sum(f2_hsum(ss2));
      if (lane == 0) {
        s_red[warp][0] = dot;
        s_red[warp][1] = ss;
      }
      __syncthreads();
      if (tid == 0) {
        float dd = 0.f, qq = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeThreads / 32; ++w) {
          dd += s_red[w][0];
          qq += s_red[w][1];
        }
        const float zp = dd * rsqrtf(fmaf(qq, p.inv_d, p.eps));
        const float lse = p.lse_inter[t];
        const float m = fmaxf(lse, zp);
        const float e1 = __expf(lse - m), e2 = __expf(zp - m);
        const float inv = __fdividef(1.0f, e1 + e2);
        s_c[0] = e1 * inv;
        s_c[1] = e2 * inv;
      }
      __syncthreads();
      c1 = s_c[0];
      c2 = s_c[1];
    }
    const uint64_t c1p = f2_pack(c1, c1), c2p = f2_pack(c2, c2);
    char* orow = p.out_r + t * row_bytes;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int v = tid + k * kMergeThreads;
      if (v < p.nvec) {
        uint64_t ri[NP];
#pragma unroll
        for (int j = 0; j < NP; j += 2) {
          const float4 f4 = *reinterpret_cast<const float4*>(rrow + v * EPV + 2 * j);
          ri[j] = f2_pack(f4.x, f4.y);
          ri[j + 1] = f2_pack(f4.z, f4.w);
        }
        uint64_t h[NP];
        if (has_p) Vec<Tin>::pairs(x[k], h);
        float out[EPV];
#pragma unroll
        for (int j = 0; j < NP; ++j) {
          uint64_t r = f2_fma(c1p, ri[j], 0);
          if (has_p) r = f2_fma(c2p, h[j], r);
          f2_unpack(r, out[2 * j], out[2 * j + 1]);
        }
        store_out<Tin, EPV>(orow, v, out);
      }
    }
    if (p.out_a && warp == 0) {
      const int na = p.n + (has_p ? 1 : 0);
      for (int s = lane; s < p.n; s += 32)
        p.out_a[t * na + s] = (p.a_inter ? p.a_inter[t * p.n + s] : 0.f) * c1;
      if (has_p && lane == 0) p.out_a[t * na + p.n] = c2;
    }
    __syncthreads();  // s_red / s_c are reused by the next token
  }
}

// The merge of a block's later layers (i >= 2) with the TMA ring, for bf16
// rows of exactly 2 x 448 16-byte vectors (d = 7168).  Per token the
// producer streams [prev (PREV), F, the fp32 inter-block row's two halves]
// into the ring; each consumer thread folds its two vectors of F into the
// partial sum (one rounding, stored), takes their dot product with w and
// their sum of squares, and after one barrier every warp forms the merge
// coefficients and writes r = c1 r_inter + c2 p.
struct MergeRingParams {
  RingParams rp;         // ring geometry; rp.T, rp.d, rp.nvec, rp.row_bytes, rp.w, rp.eps, rp.inv_d
  MergeParams mp;        // the merge's rows and outputs
};

// The merge's producer: per token the rows [prev,] F, r_inter's two halves
// into consecutive slots.  It waits for the previous kernel (pdl_wait)
// before its first row, or, with early_loads, before the first token's F
// only: prev and r_inter were written two or more launches back (see
// ring_produce), so their copies for the first token go out before the
// wait, into their own slots.
// The merge's producer: per token the rows [prev,] F, r_inter's two halves
// into consecutive slots.  It waits for the previous kernel (pdl_wait)
// before its first row, or, with early_loads, before the first token's F
// only: prev and r_inter were written two or more launches back (see
// ring_produce), so their copies for the first token go out before the
// wait, into their own slots (all on the ring's first lap, whose empty
// barriers never hold a wait).
template <bool PREV>
__device__ __forceinline__ void merge_produce(const MergeRingParams& q, RingShared& sh, uint32_t ring) {
  const RingParams& p = q.rp;
  const int nslots = p.nslots;
  const int rows = (PREV ? 1 : 0) + 1 + 2;
  const int f_row = rows - 3;
  long long issued = 0;  // rows armed, in ring order
  bool ok = true, waited = false;
  for (long long t = blockIdx.x; t < p.T && ok; t += gridDim.x) {
    const long long off = t * (long long)p.row_bytes;
    const bool early = p.early_loads && !waited;
    // pass 0 (early only): the rows not from the previous kernel; pass 1: the rest
    int armed = 0;
    for (int pass = early ? 0 : 1; pass < 2 && ok; ++pass) {
      if (pass == 1 && !waited) {
        pdl_wait();
        pdl_trigger();
        waited = true;
      }
      for (int j = 0; j < rows; ++j) {
        if (pass == 0 ? j == f_row : (early && j != f_row)) continue;
        const long long pos = issued + j;  // the row's place in ring order
        const uint32_t s = (uint32_t)(pos % nslots), l = (uint32_t)(pos / nslots);
        const char* g;
        if (PREV && j == 0) g = q.mp.prev + off;
        else if (j == f_row) g = q.mp.F + off;
        else g = reinterpret_cast<const char*>(q.mp.r_inter) + 2 * off + (j - (rows - 2)) * (long long)p.row_bytes;
        if (!mbar_wait_bounded(smem_addr(&sh.empty[s]), (l & 1u) ^ 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        const uint32_t full = smem_addr(&sh.full[s]);
        mbar_arrive_expect_tx(full, (uint32_t)p.row_bytes);
        // the bounded-wait test arms one row of the first token without its copy
        if (pos + 1 != p.withhold_row1) bulk_copy_g2s(ring + s * (uint32_t)p.row_bytes, g, (uint32_t)p.row_bytes, full);
        ++armed;
      }
    }
    // rows are armed in ring order except for the early token, where all
    // of them are (its waits cannot run out): either way the first `armed`
    // positions of this token hold every copy issued
    issued += armed;
  }
  if (!waited) {
    pdl_wait();
    pdl_trigger();
  }
  if (!ok) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
  ring_drain(sh.full, nslots, issued, p.withhold_row1);
}

template <bool PREV>
__global__ void __launch_bounds__(kRingThreads, 1) agg_merge_ring_kernel(const __grid_constant__ MergeRingParams q) {
  const RingParams& p = q.rp;
  const MergeParams& mp = q.mp;
  extern __shared__ __align__(128) unsigned char smem[];
  RingShared& sh = *reinterpret_cast<RingShared*>(smem);
  const uint32_t ring = smem_addr(smem) + kRingHeaderBytes;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nslots = p.nslots;
  ring_init(p, sh);
  __syncthreads();
  if (warp == kRingConsumerWarps) {
    // the producer waits for the previous kernel itself (early loads)
    if (lane == 0) merge_produce<PREV>(q, sh, ring);
    pdl_wait();
    pdl_trigger();
    return;
  }
  pdl_wait();
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done

  uint64_t wp[2][4];  // this thread's channels of w (vectors tid, tid + 448), as pairs
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int v = tid + k * kRingConsumers;
#pragma unroll
    for (int j = 0; j < 4; ++j) wp[k][j] = f2_pack(__ldg(p.w + v * 8 + 2 * j), __ldg(p.w + v * 8 + 2 * j + 1));
  }
  const long long T = p.T;
  const float nan = __int_as_float(0x7fc00000);
  uint32_t slot = 0, lap = 0;
  bool ok = true;
  int iter = 0;
  bool abort = false;
  // take 32 bytes per thread of the next slot: a bf16 row's vectors tid and
  // tid + 448 (halves = false), or one fp32 half row's bytes [32 tid, +32)
  auto consume = [&](uint4* dst, bool halves) {
    if (ok && !mbar_wait_bounded_sh(smem_addr(&sh.full[slot]), lap & 1u, &sh.wait_ns)) ok = false;
    const uint32_t base = ring + slot * (uint32_t)p.row_bytes;
    if (halves) {
      dst[0] = ld_shared_v4(base + (uint32_t)tid * 32u);
      dst[1] = ld_shared_v4(base + (uint32_t)tid * 32u + 16u);
    } else {
      dst[0] = ld_shared_v4(base + (uint32_t)tid * 16u);
      dst[1] = ld_shared_v4(base + (uint32_t)(tid + kRingConsumers) * 16u);
    }
    // Lane 0 releases the slot only while its own waits have all succeeded
    // (the safe abort protocol of the ring kernels).
    __syncwarp();
    if (lane == 0 && ok) mbar_arrive(smem_addr(&sh.empty[slot]));
    if (++slot == (uint32_t)nslots) {
      slot = 0;
      ++lap;
    }
  };

  for (long long t = blockIdx.x; t < T && !abort; t += gridDim.x, ++iter) {
    const int buf = iter & 1;
    volatile int* abort_flag = &sh.abort_flag[buf];
    const float lse = __ldg(mp.lse_inter + t);
    uint4 pv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)}, fv[2];
    if (PREV) consume(pv, false);
    consume(fv, false);
    // the new partial sum: prev + F, rounded once, stored
    uint4 x[2];
    char* drow = mp.dst + t * (long long)p.row_bytes;
    uint64_t dot2 = 0, ss2 = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      float f[8];
      Vec<bf16_t>::unpack(fv[k], f);
      if (PREV) {
        float g[8];
        Vec<bf16_t>::unpack(pv[k], g);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = g[e] + f[e];
      }
      if (!ok) {
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = nan;
      }
      x[k] = Vec<bf16_t>::pack(f);
      *reinterpret_cast<uint4*>(drow + (size_t)(tid + k * kRingConsumers) * 16) = x[k];
      uint64_t h[4];
      Vec<bf16_t>::pairs(x[k], h);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        dot2 = f2_fma(wp[k][j], h[j], dot2);
        ss2 = f2_fma(h[j], h[j], ss2);
      }
    }
    const float dot = warp_sum(f2_hsum(dot2)), ss = warp_sum(f2_hsum(ss2));
    if (lane == 0) {
      sh.red[buf][warp][0] = dot;
      sh.red[buf][warp][1] = ss;
    }
    // the fp32 inter-block row: thread tid's vectors' 32 bytes in each half
    uint4 r0[2], r1[2];
    consume(r0, true);
    consume(r1, true);
    const bool warp_failed = __any_sync(0xffffffffu, !ok);
    if (lane == 0 && warp_failed) *abort_flag = 1;
    named_barrier_sync(kRingBarrierId, kRingConsumers);
    abort = *abort_flag != 0;

    float c1 = nan, c2 = nan;
    if (!abort) {
      float dd = 0.f, qq = 0.f;
#pragma unroll
      for (int w = 0; w < kRingConsumerWarps; ++w) {
        dd += sh.red[buf][w][0];
        qq += sh.red[buf][w][1];
      }
      // fast reciprocal square root, exponential and division: a few fp32
      // ulps, far inside the parity tolerances
      const float zp = dd * rsqrtf(fmaf(qq, p.inv_d, p.eps));
      const float m = fmaxf(lse, zp);
      const float e1 = __expf(lse - m), e2 = __expf(zp - m);
      const float inv = __fdividef(1.0f, e1 + e2);
      c1 = e1 * inv;
      c2 = e2 * inv;
    }
    const uint64_t c1p = f2_pack(c1, c1), c2p = f2_pack(c2, c2);
    char* orow = mp.out_r + t * (long long)p.row_bytes;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4* rr = k == 0 ? r0 : r1;
      uint64_t ri[4] = {f2_pack(__uint_as_float(rr[0].x), __uint_as_float(rr[0].y)),
                        f2_pack(__uint_as_float(rr[0].z), __uint_as_float(rr[0].w)),
                        f2_pack(__uint_as_float(rr[1].x), __uint_as_float(rr[1].y)),
                        f2_pack(__uint_as_float(rr[1].z), __uint_as_float(rr[1].w))};
      uint64_t h[4];
      Vec<bf16_t>::pairs(x[k], h);
      float out[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t r = f2_fma(c2p, h[j], f2_fma(c1p, ri[j], 0));
        f2_unpack(r, out[2 * j], out[2 * j + 1]);
      }
      store_out<bf16_t, 8>(orow, tid + k * kRingConsumers, out);
    }
    if (mp.out_a && warp == 0) {
      const int na = mp.n + 1;
      for (int s2 = lane; s2 < mp.n; s2 += 32)
        mp.out_a[t * na + s2] = (mp.a_inter ? __ldg(mp.a_inter + t * mp.n + s2) : 0.f) * c1;
      if (lane == 0) mp.out_a[t * na + mp.n] = c2;
    }
    if (abort && tid == 0) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
  }
}

// ---------------------------------------------------------------- launch --

template <typename Tin, int VPT, bool EXACT, bool DOTS = false, int NS = 0>
static cudaError_t launch_inter_t(const InterParams& ip, int grid, int smem, cudaStream_t stream) {
  static SmemOptIn optin;  // the large shared-memory opt-in, per device and context
  auto kern = [] {
    if constexpr (DOTS)
      return agg_interblock_dots_kernel<2 * VPT, EXACT, NS>;  // bf16 rows: two quads per 16-byte vector
    else
      return agg_interblock_kernel<Tin, VPT, EXACT>;
  }();
  cudaError_t e = optin.ensure(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  e = launch_kernel(kern, dim3(grid), dim3(kRingThreads), (size_t)smem, stream, ip);
  return e != cudaSuccess ? e : cudaGetLastError();
}

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Geometry both phases need: 16-byte rows of at most 2 x 448 vectors.
static bool twophase_geometry(int d, int dtype, int* nvec, int* vpt) {
  const int esz = dtype == ATTNRES_BF16 ? 2 : 4;
  const long long row_bytes = (long long)d * esz;
  if (row_bytes % 16 != 0) return false;
  *nvec = (int)(row_bytes / 16);
  *vpt = (*nvec + kRingConsumers - 1) / kRingConsumers;
  return *vpt >= 1 && *vpt <= kRingMaxVpt;
}

bool twophase_supported(int d, int dtype) {
  int nvec, vpt;
  return twophase_geometry(d, dtype, &nvec, &vpt);
}

cudaError_t launch_interblock(const InterArgs& a) {
  if (a.T <= 0) return cudaSuccess;
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  int nvec = 0, vpt = 0;
  if (!twophase_geometry(a.d, a.dtype, &nvec, &vpt)) return cudaErrorInvalidValue;
  const bool bf16 = a.dtype == ATTNRES_BF16;
  const int row_bytes = nvec * 16;
  InterParams ip{};
  RingParams& rp = ip.rp;
  for (int s = 0; s < a.n; ++s) rp.src[s] = static_cast<const char*>(a.src[s]);
  rp.w = a.wq[0];
  rp.dev_err = a.dev_err;
  rp.T = a.T;
  rp.d = a.d;
  rp.n_stored = a.n;
  rp.S = a.n;
  rp.nvec = nvec;
  rp.row_bytes = row_bytes;
  rp.out_row_bytes = a.d * 4;
  rp.eps = a.eps;
  rp.inv_d = 1.0f / (float)a.d;
  rp.wait_ns = wait_limit_ns();
  rp.withhold_row1 = debug_withhold_row1();
  // the one-pass kernel keeps a token's n rows in the ring until it is done:
  // the ring must hold them
  int nslots = (di.max_smem_optin - kRingHeaderBytes - kInterSharedBytes) / row_bytes;
  if (nslots > kRingMaxSlots) nslots = kRingMaxSlots;
  if (nslots < a.n) return cudaErrorInvalidValue;
  rp.nslots = nslots;
  for (int q = 0; q < a.Q; ++q) ip.wq[q] = a.wq[q];
  ip.Q = a.Q;
  ip.out_r = a.out_r;
  ip.out_lse = a.out_lse;
  ip.out_a = a.out_a;
  ip.out_r0 = static_cast<char*>(a.out_r0);
  ip.out_a0 = a.out_a0;
  int grid = (int)(a.T < di.sm_count ? a.T : di.sm_count);
  const int smem = kRingHeaderBytes + kInterSharedBytes + nslots * row_bytes;
  const bool exact = nvec == vpt * kRingConsumers;
  if (a.workspace && interblock_tc_supported(a.n, a.d, a.dtype)) {
    // the logits on the tensor cores, then the softmax and the weighted sums here
    float* dots = nullptr;
    int ksplit = 0;
    e = launch_interblock_tc(a, a.workspace, &dots, &ksplit);
    if (e != cudaSuccess) return e;
    ip.dots = dots;
    ip.ksplit = ksplit;
    // one CTA per SM; the tokens of the last, partial round split by query
    // groups over the idle CTAs (every token once when T is below the SMs)
    const int G = di.sm_count;
    const long long r = a.T % G;
    ip.tail_groups = r == 0 ? 1 : (int)(G / r < a.Q ? G / r : a.Q);
    grid = G;
    if (vpt == 1) return launch_inter_t<bf16_t, 1, false, true>(ip, grid, smem, a.stream);
    if (!exact) return launch_inter_t<bf16_t, 2, false, true>(ip, grid, smem, a.stream);
    switch (a.n) {  // d = 7168: the source count fixed at compile time
      case 1: return launch_inter_t<bf16_t, 2, true, true, 1>(ip, grid, smem, a.stream);
      case 2: return launch_inter_t<bf16_t, 2, true, true, 2>(ip, grid, smem, a.stream);
      case 3: return launch_inter_t<bf16_t, 2, true, true, 3>(ip, grid, smem, a.stream);
      case 4: return launch_inter_t<bf16_t, 2, true, true, 4>(ip, grid, smem, a.stream);
      case 5: return launch_inter_t<bf16_t, 2, true, true, 5>(ip, grid, smem, a.stream);
      case 6: return launch_inter_t<bf16_t, 2, true, true, 6>(ip, grid, smem, a.stream);
      case 7: return launch_inter_t<bf16_t, 2, true, true, 7>(ip, grid, smem, a.stream);
      case 8: return launch_inter_t<bf16_t, 2, true, true, 8>(ip, grid, smem, a.stream);
      default: return launch_inter_t<bf16_t, 2, true, true, 9>(ip, grid, smem, a.stream);
    }
  }
  if (bf16) {
    if (vpt == 1) return launch_inter_t<bf16_t, 1, false>(ip, grid, smem, a.stream);
    return exact ? launch_inter_t<bf16_t, 2, true>(ip, grid, smem, a.stream)
                 : launch_inter_t<bf16_t, 2, false>(ip, grid, smem, a.stream);
  }
  if (vpt == 1) return launch_inter_t<float, 1, false>(ip, grid, smem, a.stream);
  return exact ? launch_inter_t<float, 2, true>(ip, grid, smem, a.stream)
               : launch_inter_t<float, 2, false>(ip, grid, smem, a.stream);
}

template <bool PREV>
static cudaError_t launch_merge_ring_t(const MergeRingParams& q, int grid, int smem, cudaStream_t stream) {
  static SmemOptIn optin;  // the large shared-memory opt-in, per device and context
  auto kern = agg_merge_ring_kernel<PREV>;
  cudaError_t e = optin.ensure(reinterpret_cast<const void*>(kern));
  if (e != cudaSuccess) return e;
  e = launch_kernel(kern, dim3(grid), dim3(kRingThreads), (size_t)smem, stream, q);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs& a) {
  if (a.T <= 0) return cudaSuccess;
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  int nvec = 0, vpt = 0;
  if (!twophase_geometry(a.d, a.dtype, &nvec, &vpt)) return cudaErrorInvalidValue;
  if (a.F && a.dtype == ATTNRES_BF16 && nvec == 2 * kRingConsumers) {
    // a later layer of the block, bf16 rows of 2 x 448 vectors: the ring
    MergeRingParams q{};
    RingParams& rp = q.rp;
    rp.w = a.w;
    rp.T = a.T;
    rp.d = a.d;
    rp.nvec = nvec;
    rp.row_bytes = nvec * 16;
    rp.eps = a.eps;
    rp.inv_d = 1.0f / (float)a.d;
    rp.wait_ns = wait_limit_ns();
    rp.withhold_row1 = debug_withhold_row1();
    rp.early_loads = a.early_loads ? 1 : 0;
    rp.dev_err = a.dev_err;
    int nslots = (di.max_smem_optin - kRingHeaderBytes) / rp.row_bytes;
    if (nslots > kRingMaxSlots) nslots = kRingMaxSlots;
    if (nslots < 4) return cudaErrorInvalidValue;
    rp.nslots = nslots;
    MergeParams& mp = q.mp;
    mp.prev = static_cast<const char*>(a.prev);
    mp.F = static_cast<const char*>(a.F);
    mp.dst = static_cast<char*>(a.dst);
    mp.w = a.w;
    mp.r_inter = a.r_inter;
    mp.lse_inter = a.lse_inter;
    mp.a_inter = a.a_inter;
    mp.out_r = static_cast<char*>(a.out_r);
    mp.out_a = a.out_a;
    mp.T = a.T;
    mp.d = a.d;
    mp.n = a.n;
    mp.nvec = nvec;
    mp.eps = a.eps;
    mp.inv_d = rp.inv_d;
    const int grid = (int)(a.T < di.sm_count ? a.T : di.sm_count);
    const int smem = kRingHeaderBytes + nslots * rp.row_bytes;
    return a.prev ? launch_merge_ring_t<true>(q, grid, smem, a.stream) : launch_merge_ring_t<false>(q, grid, smem, a.stream);
  }
  MergeParams mp{};
  mp.prev = static_cast<const char*>(a.prev);
  mp.F = static_cast<const char*>(a.F);
  mp.dst = static_cast<char*>(a.dst);
  mp.w = a.w;
  mp.r_inter = a.r_inter;
  mp.lse_inter = a.lse_inter;
  mp.a_inter = a.a_inter;
  mp.out_r = static_cast<char*>(a.out_r);
  mp.out_a = a.out_a;
  mp.T = a.T;
  mp.d = a.d;
  mp.n = a.n;
  mp.nvec = nvec;
  mp.eps = a.eps;
  mp.inv_d = 1.0f / (float)a.d;
  const long long cap = (long long)di.sm_count * 4;
  const int grid = (int)(a.T < cap ? a.T : cap);
  const bool bf16 = a.dtype == ATTNRES_BF16;
  if (bf16) {
    e = vpt == 1 ? launch_kernel(agg_merge_kernel<bf16_t, 1>, dim3(grid), dim3(kMergeThreads), 0, a.stream, mp)
                 : launch_kernel(agg_merge_kernel<bf16_t, 2>, dim3(grid), dim3(kMergeThreads), 0, a.stream, mp);
  } else {
    e = vpt == 1 ? launch_kernel(agg_merge_kernel<float, 1>, dim3(grid), dim3(kMergeThreads), 0, a.stream, mp)
                 : launch_kernel(agg_merge_kernel<float, 2>, dim3(grid), dim3(kMergeThreads), 0, a.stream, mp);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

bool twophase_pointers_ok(const void* p) { return p == nullptr || al16(p); }

}  // namespace attnres
