// The logits of the two-phase schedule's inter-block pass on the tensor
// cores (Kimi K3 chaptered tutorial, ch. 4.4 and 4.6: one batched pass over
// the cached block sums for all of a block's layer queries).
//
// For a block with n cached sources and Q layer queries, every token t needs
// the Q x n dot products w_q . h_s[t].  Over all tokens they form one dense
// product, (T n rows of d) x (d x Q), in which every token shares the same
// queries: on the CUDA cores each token would stream the queries again.
// Here a tile of tt tokens x n sources (128 rows, each source's tt rows one
// TMA tensor box) is multiplied on the tensor cores against the queries,
// which are read once per tile.
//
// interblock_dots_kernel: tcgen05.mma kind::f16 (bf16 in, fp32 accumulate
// in TMEM), M = 128 rows, N = 48, K = 16 per instruction, 64 channels per
// pipeline stage.  The queries enter as three bf16 terms, w_q (fp32) =
// hi + mid + lo, so that bf16 x bf16 products summed in fp32 keep the fp32
// query's precision: rows 16 j + q of the stage's B tile (term j, query q;
// rows q >= Q zero).  Warp 0 issues the TMA loads of the source rows,
// warp 1 the MMAs; warps 2-5 first write each stage's B tile (the query
// split, from the fp32 queries, in the layout the TMA would give), then read
// the accumulator back (tcgen05.ld) and store hi + mid + lo per query.  The
// channels are split across CTAs (split-K) so that every SM has work; each
// split writes its own partial dots.
//
// The softmax, the log-sum-exp and the weighted sums follow in
// agg_interblock_dots_kernel (twophase.cu), which sums the partial dots in a
// fixed order.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "ring_common.cuh"

namespace attnres {

constexpr int kTcRows = 128;                           // M: tt tokens x np sources
constexpr int kTcN = 48;                               // 3 terms x 16 query rows
constexpr int kTcChunk = 64;                           // channels per stage: one 128-byte swizzle row
constexpr int kTcABytes = kTcRows * 128;               // 16 KB
constexpr int kTcBBytes = kTcN * 128;                  // 6 KB
constexpr int kTcStageBytes = kTcABytes + kTcBBytes;   // 22 KB, a multiple of 1024
constexpr int kTcStages = 4;
constexpr int kTcThreads = 192;                        // 6 warps
constexpr int kTcTmemCols = 64;                        // the 48 accumulator columns, rounded up
constexpr int kTcSmemBytes = kTcStages * kTcStageBytes + 1024;  // + alignment slack
constexpr int kTcMaxSplit = 16;                        // channel splits per tile, at most (kInterMaxSplit)

static_assert(kTcStageBytes % 1024 == 0, "stages must keep 1024-byte alignment (128-byte swizzle atoms)");

struct DotsParams {
  CUtensorMap src[kRingSmax];  // per cached source: [T, d] bf16, box {64 channels, tt tokens}, 128-byte swizzle
  InterQueries wq;             // the Q fp32 queries [d], 16-byte aligned
  float* dots;                 // [ksplit][T][n][Q] fp32 partial dot products
  long long T;
  int n, tt, Q;
  int nchunks, chunks_per_split, ksplit;
  int* dev_err;
  unsigned long long wait_ns;
};

// ---------------------------------------------------------------- PTX ------

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// one warp: allocate ncols TMEM columns, their address written to *dst (shared)
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T, both K-major bf16, fp32 accumulate
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// the mbarrier at `bar` receives one arrival once every MMA this thread
// issued so far has completed
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes (one per thread)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile stored as
// 128-byte rows in the 128-byte swizzle (as TMA writes them): start address,
// stride between 8-row groups 1024 bytes, the descriptor version of this
// architecture (bits 46-47 = 1), swizzle mode 128 B (bits 61-63 = 2).  The
// leading offset is unused for swizzled K-major tiles (1 by convention).
__device__ __forceinline__ uint64_t smem_desc_k128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kTcIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTcN >> 3) << 17) |
                              ((uint32_t)(kTcRows >> 4) << 24);

// ------------------------------------------------------------- kernels -----

// Three bf16 terms of 8 fp32 query values (channels 8 j .. 8 j + 7):
// hi = round(w), mid = round(w - hi), lo = round(w - hi - mid), each
// subtraction exact; as 16-byte rows of 8 bf16 each.
__device__ __forceinline__ void split3(const float4& a, const float4& b, uint4* hi, uint4* mid, uint4* lo) {
  const float w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t th[4], tm[4], tl[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t h = pack_bf16x2(w[2 * k], w[2 * k + 1]);
    const float r0 = w[2 * k] - bf16lo(h), r1 = w[2 * k + 1] - bf16hi(h);
    const uint32_t m = pack_bf16x2(r0, r1);
    const float s0 = r0 - bf16lo(m), s1 = r1 - bf16hi(m);
    th[k] = h;
    tm[k] = m;
    tl[k] = pack_bf16x2(s0, s1);
  }
  *hi = make_uint4(th[0], th[1], th[2], th[3]);
  *mid = make_uint4(tm[0], tm[1], tm[2], tm[3]);
  *lo = make_uint4(tl[0], tl[1], tl[2], tl[3]);
}

__global__ void __launch_bounds__(kTcThreads, 1) interblock_dots_kernel(const __grid_constant__ DotsParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full[kTcStages], bfull[kTcStages], empty[kTcStages], acc_full;
  __shared__ uint32_t tmem_base;
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1024-byte alignment
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x / p.ksplit, ks = blockIdx.x % p.ksplit;
  const long long t0 = (long long)tile * p.tt;
  const int c0 = ks * p.chunks_per_split;
  const int c1 = c0 + p.chunks_per_split < p.nchunks ? c0 + p.chunks_per_split : p.nchunks;
  const int nloc = c1 - c0;  // >= 1 (the host sizes the splits so)

  // rows n * tt .. 127 of every stage's A tile hold no source, and the B
  // tiles' rows of queries q >= Q none: zero, once (no later write touches
  // them; the tensor cores read them as zeros)
  const int used = p.n * p.tt * 128;
  for (int st = 0; st < kTcStages; ++st) {
    for (int off = used + tid * 16; off < kTcABytes; off += kTcThreads * 16)
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(base + st * kTcStageBytes + off), "r"(0)
                   : "memory");
    for (int off = tid * 16; off < kTcBBytes; off += kTcThreads * 16)
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(base + st * kTcStageBytes + kTcABytes + off),
                   "r"(0)
                   : "memory");
  }
  fence_proxy_async_smem();  // those generic stores, before the tensor cores read the tiles
  if (tid == 0) {
    for (int st = 0; st < kTcStages; ++st) {
      mbar_init(smem_addr(&full[st]), 1);
      mbar_init(smem_addr(&bfull[st]), kTcThreads / 32 - 2);  // one arrival per warp of warps 2-5
      mbar_init(smem_addr(&empty[st]), 1);
    }
    mbar_init(smem_addr(&acc_full), 1);
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(&tmem_base), kTcTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  pdl_wait();  // the sources and the queries may come from the previous kernels
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done

  if (warp == 0) {
    if (lane == 0) {
      // producer: the tile's n boxes of tt rows, per stage
      const uint32_t tx = (uint32_t)(p.n * p.tt * 128);
      int issued = 0;
      for (int i = 0; i < nloc; ++i) {
        const int st = i % kTcStages;
        const uint32_t lap = (uint32_t)(i / kTcStages);
        if (!mbar_wait_bounded(smem_addr(&empty[st]), (lap & 1u) ^ 1u, p.wait_ns)) {
          report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
          break;
        }
        const uint32_t fb = smem_addr(&full[st]);
        mbar_arrive_expect_tx(fb, tx);
        const int x = (c0 + i) * kTcChunk;
        const uint32_t a = base + st * kTcStageBytes;
        for (int s = 0; s < p.n; ++s) tma_load_2d(a + s * p.tt * 128, &p.src[s], x, (int)t0, fb);
        ++issued;
      }
      // the CTA never exits under a copy: wait for the latest phase of every
      // stage that received one
      const int armed = issued < kTcStages ? issued : kTcStages;
      for (int st = 0; st < armed; ++st) {
        const int uses = (issued - 1 - st) / kTcStages + 1;
        mbar_wait_bounded(smem_addr(&full[st]), (uint32_t)((uses - 1) & 1));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer: 4 instructions of K = 16 per 64-channel stage
      for (int i = 0; i < nloc; ++i) {
        const int st = i % kTcStages;
        const uint32_t lap = (uint32_t)(i / kTcStages);
        if (!mbar_wait_bounded(smem_addr(&full[st]), lap & 1u, p.wait_ns) ||
            !mbar_wait_bounded(smem_addr(&bfull[st]), lap & 1u, p.wait_ns)) {
          report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t a = base + st * kTcStageBytes, b = a + kTcABytes;
#pragma unroll
        for (int kk = 0; kk < kTcChunk / 16; ++kk)
          tc_mma_bf16(tmem, smem_desc_k128(a + kk * 32), smem_desc_k128(b + kk * 32), kTcIdesc,
                      (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(smem_addr(&empty[st]));  // the stage is free once these MMAs have read it
      }
      tc_commit(smem_addr(&acc_full));  // the accumulator is final once every MMA above is done
    }
    __syncwarp();
  } else {
    // the queries' B tiles: thread i writes 16 bytes (channels 8 bj .. + 7,
    // bj = i mod 8) of query bq = i / 8 into rows bq, 16 + bq, 32 + bq, at
    // the 128-byte swizzle's position of that chunk (bj ^ row mod 8).  Its
    // loads run kTcStages chunks ahead (an L2 round trip is longer than a
    // stage).
    const int bi = tid - 64, bq = bi >> 3, bj = bi & 7;
    const bool act = bq < p.Q;
    const float4* wsrc = reinterpret_cast<const float4*>(act ? p.wq.w[bq] + c0 * kTcChunk + 8 * bj : nullptr);
    constexpr int kPf = kTcStages;
    float4 wa[kPf], wb[kPf];
#pragma unroll
    for (int u = 0; u < kPf; ++u) {
      wa[u] = wb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (act && u < nloc) {
        wa[u] = __ldg(wsrc + u * (kTcChunk / 4));
        wb[u] = __ldg(wsrc + u * (kTcChunk / 4) + 1);
      }
    }
    bool bok = true;
    for (int i0 = 0; i0 < nloc && bok; i0 += kPf) {
#pragma unroll
      for (int u = 0; u < kPf; ++u) {
        const int i = i0 + u;
        if (i < nloc && bok) {
          const int st = i % kTcStages;
          const uint32_t lap = (uint32_t)(i / kTcStages);
          // warp-uniform outcome: the warp arrives once, after all its lanes wrote
          if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&empty[st]), (lap & 1u) ^ 1u, p.wait_ns))) {
            if (lane == 0) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
            bok = false;
          } else {
            if (act) {
              uint4 th, tm, tl;
              split3(wa[u], wb[u], &th, &tm, &tl);
              const uint32_t bt = base + st * kTcStageBytes + kTcABytes;
              const uint4* terms[3] = {&th, &tm, &tl};
#pragma unroll
              for (int term = 0; term < 3; ++term) {
                const int row = 16 * term + bq;
                const uint4 v = *terms[term];
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(bt + row * 128 + ((bj ^ (row & 7)) << 4)),
                             "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                             : "memory");
              }
              if (i + kPf < nloc) {
                wa[u] = __ldg(wsrc + (i + kPf) * (kTcChunk / 4));
                wb[u] = __ldg(wsrc + (i + kPf) * (kTcChunk / 4) + 1);
              }
            }
            fence_proxy_async_smem();  // visible to the tensor cores
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bfull[st]));
          }
        }
      }
    }

    // epilogue: warp w reads TMEM lanes 32 (w mod 4) .. + 31, one row per thread
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&acc_full), 0u, p.wait_ns));
    if (!ok && lane == 0) report_error(p.dev_err, ATTNRES_DEVERR_WAIT_TIMEOUT);
    tc_fence_after();  // the warp is converged here for the .sync.aligned loads
    const int g = warp & 3;
    uint32_t v[kTcN];
    const uint32_t taddr = tmem + ((uint32_t)(32 * g) << 16);
    tmem_ld16(taddr + 0, v);
    tmem_ld16(taddr + 16, v + 16);
    tmem_ld16(taddr + 32, v + 32);
    tmem_ld_wait();
    const int row = 32 * g + lane;
    const int s = row / p.tt, j = row % p.tt;
    const long long t = t0 + j;
    if (s < p.n && t < p.T) {
      float* out = p.dots + (((long long)ks * p.T + t) * p.n + s) * p.Q;
      const float nan = __int_as_float(0x7fc00000);
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (q < p.Q)
          out[q] = ok ? (__uint_as_float(v[q]) + __uint_as_float(v[16 + q])) + __uint_as_float(v[32 + q]) : nan;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

// ---------------------------------------------------------------- host -----

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(f);
  });
  return fn;
}

// a [rows, d] bf16 row-major matrix, boxes of {64 channels, box_rows rows}
bool make_map(CUtensorMap* map, const void* ptr, long long rows, int d, int box_rows) {
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTcChunk, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcGeometry {
  int tt, ntiles, nchunks, chunks_per_split, ksplit;
  long long dots_bytes;
};

// tt tokens per tile (n sources each, n rounded up to a power of two so
// that tt * np = 128); the channel range split so that the tiles' CTAs fill
// the two CTA slots of every SM once.
TcGeometry tc_geometry(int n, long long T, int d, int Q, int sm_count) {
  TcGeometry g{};
  int np = 1;
  while (np < n) np *= 2;
  g.tt = kTcRows / np;
  g.ntiles = (int)((T + g.tt - 1) / g.tt);
  g.nchunks = d / kTcChunk;
  // two CTAs fit on an SM: one wave of 2 x SMs CTAs (a second, partial wave
  // would idle most SMs while it runs)
  const long long slots = 2LL * sm_count;
  long long ks = slots / g.ntiles;
  if (ks < 1) ks = 1;
  if (ks > kTcMaxSplit) ks = kTcMaxSplit;  // the softmax sums this many partials per logit
  if (ks > g.nchunks) ks = g.nchunks;
  g.chunks_per_split = (int)((g.nchunks + ks - 1) / ks);
  g.ksplit = (g.nchunks + g.chunks_per_split - 1) / g.chunks_per_split;  // every split has >= 1 chunk
  g.dots_bytes = (long long)g.ksplit * T * n * Q * 4;
  return g;
}

long long align256(long long x) { return (x + 255) & ~255LL; }

}  // namespace

bool interblock_tc_supported(int n, int d, int dtype) {
  return dtype == ATTNRES_BF16 && d % kTcChunk == 0 && n >= 1 && n <= kRingSmax && encode_fn() != nullptr;
}

int64_t interblock_tc_workspace_bytes(int n, long long T, int d, int dtype, int Q) {
  if (!interblock_tc_supported(n, d, dtype) || T <= 0) return 0;
  DeviceInfo di;
  if (device_info(&di) != cudaSuccess) return -1;
  const TcGeometry g = tc_geometry(n, T, d, Q, di.sm_count);
  return align256(g.dots_bytes);
}

namespace {
thread_local const char* g_tc_step = "";
// a refused launch also leaves its error as the runtime's last error: clear
// it, so that the next call's launch check does not see it again
cudaError_t tc_fail(cudaError_t e, const char* step) {
  g_tc_step = step;
  (void)cudaGetLastError();
  return e;
}
}  // namespace

const char* interblock_tc_last_step() { return g_tc_step; }

cudaError_t launch_interblock_tc(const InterArgs& a, void* workspace, float** dots_out, int* ksplit_out) {
  g_tc_step = "";
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return tc_fail(e, "device query");
  const TcGeometry g = tc_geometry(a.n, a.T, a.d, a.Q, di.sm_count);
  float* dots = static_cast<float*>(workspace);

  DotsParams dp{};
  for (int s = 0; s < a.n; ++s)
    if (!make_map(&dp.src[s], a.src[s], a.T, a.d, g.tt)) return tc_fail(cudaErrorInvalidValue, "source tensor map");
  for (int q = 0; q < a.Q; ++q) dp.wq.w[q] = a.wq[q];
  dp.dots = dots;
  dp.T = a.T;
  dp.n = a.n;
  dp.tt = g.tt;
  dp.Q = a.Q;
  dp.nchunks = g.nchunks;
  dp.chunks_per_split = g.chunks_per_split;
  dp.ksplit = g.ksplit;
  dp.dev_err = a.dev_err;
  dp.wait_ns = wait_limit_ns();
  static SmemOptIn optin;
  e = optin.ensure(reinterpret_cast<const void*>(interblock_dots_kernel), kTcSmemBytes);
  if (e != cudaSuccess) return tc_fail(e, "shared-memory opt-in");
  e = launch_kernel(interblock_dots_kernel, dim3(g.ntiles * g.ksplit), dim3(kTcThreads), (size_t)kTcSmemBytes,
                    a.stream, dp);
  if (e != cudaSuccess) return tc_fail(e, "logits launch");
  *dots_out = dots;
  *ksplit_out = g.ksplit;
  return cudaSuccess;
}

}  // namespace attnres
