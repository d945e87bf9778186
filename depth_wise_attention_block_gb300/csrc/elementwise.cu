// Elementwise kernels of the stack:
//
//  fold_kernel        the block bookkeeping on its own (Kimi K3 chaptered
//                     tutorial, ch. 4.3 Eq. 10 and ch. 4.6): the output v of
//                     a layer is added to the running partial sum of its
//                     block, dst = round(prev + v), or copied when the
//                     partial sum is empty.  The fused path of the ring kernel (ring_kernel.cuh)
//                     does the same arithmetic inside the aggregation.
//  synth_layer_kernel the stand-in layer body F(x) = tanh(x * g) * s used to
//                     drive a stack without trained weights.
//  synth_layer_backward_kernel  its gradient, dx = (dv_a + dv_b) *
//                     sech(x g)^2 * g * s (dv_b optional).
//
// Both are HBM-bound streams: 16-byte vector accesses when every pointer is
// 16-byte aligned and rows hold whole vectors, scalar accesses otherwise;
// grid-stride loops over a grid sized to the SM count.
#include <math.h>

#include "attnres.h"
#include "device_common.cuh"
#include "launch.h"

namespace attnres {

constexpr int kEwThreads = 256;
constexpr int kEwCtasPerSm = 8;  // 2048 threads per SM

template <typename T>
struct Vec16;
template <>
struct Vec16<bf16_t> {
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
};
template <>
struct Vec16<float> {
  static constexpr int kElems = 4;
  static __device__ __forceinline__ void unpack(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ uint4 pack(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

// ------------------------------------------------------------------ fold --

template <typename T, bool VEC>
__global__ void __launch_bounds__(kEwThreads) fold_kernel(const T* prev, const T* F, T* dst,
                                                          long long n) {
  // dst may alias prev (the partial sum is updated in place)
  pdl_wait();
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done
  const long long stride = (long long)gridDim.x * blockDim.x;
  if constexpr (VEC) {
    constexpr int E = Vec16<T>::kElems;
    const long long nv = n / E;
    const uint4* F4 = reinterpret_cast<const uint4*>(F);
    const uint4* P4 = reinterpret_cast<const uint4*>(prev);
    uint4* D4 = reinterpret_cast<uint4*>(dst);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
      float f[E];
      Vec16<T>::unpack(F4[i], f);
      if (prev) {
        float q[E];
        Vec16<T>::unpack(P4[i], q);
#pragma unroll
        for (int e = 0; e < E; ++e) f[e] = q[e] + f[e];
      }
      D4[i] = Vec16<T>::pack(f);
    }
  } else {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
      float x = load_elem(F + i);
      if (prev) x = load_elem(prev + i) + x;
      store_elem(dst + i, x);
    }
  }
}

// ------------------------------------------------------- synthetic layer --

// tanh of the stand-in body.  With bf16 storage it is the hardware
// approximation (tanh.approx.f32, relative error about 2^-11 by the PTX ISA):
// below half a bf16 ulp (2^-9 relative), so a stored value moves by at most
// one ulp, and only where the exact value lies next to a rounding boundary;
// tanhf costs enough instructions to hold an L2-warm layer body to ~60 % of
// the copy rate.  fp32 storage keeps tanhf.
template <typename T>
__device__ __forceinline__ float body_tanh(float x);
template <>
__device__ __forceinline__ float body_tanh<bf16_t>(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
template <>
__device__ __forceinline__ float body_tanh<float>(float x) {
  return tanhf(x);
}

// sech^2(u) = 1 - tanh(u)^2, the derivative of tanh, for the gradient of the
// stand-in body.  From one exponential: with E = exp(-2|u|) in (0, 1],
// sech^2(u) = 4E / (1 + E)^2.  Every term is positive, so nothing cancels
// (1 - tanh^2 loses the relative precision of its small values where |tanh|
// nears 1); the fast exponential's relative error grows like |u| 2^-23,
// a few fp32 ulps where sech^2 is not negligible.
__device__ __forceinline__ float sech2(float u) {
  const float E = __expf(-2.f * fabsf(u));
  const float q = 1.f + E;
  return __fdividef(4.f * E, q * q);
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kEwThreads) synth_layer_kernel(const T* x, const float* __restrict__ g,
                                                                 const float* __restrict__ s, T* out,
                                                                 long long T_, int d) {
  pdl_wait();
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done
  const long long n = T_ * (long long)d;
  const long long stride = (long long)gridDim.x * blockDim.x;
  if constexpr (VEC) {
    // A thread owns one 16-byte channel vector (its g and s stay in
    // registers) and walks down the tokens, kUnroll rows in flight at a
    // time; consecutive threads take consecutive vectors of a row.
    constexpr int E = Vec16<T>::kElems;
    constexpr int kUnroll = 4;
    const int vrow = d / E;  // vectors per row (d % E == 0 here)
    const int cv = blockIdx.x * blockDim.x + threadIdx.x;
    if (cv < vrow) {
      float gg[E], ss[E];
#pragma unroll
      for (int e = 0; e < E; e += 4) {
        const float4 g4 = __ldg(reinterpret_cast<const float4*>(g + cv * E + e));
        const float4 s4 = __ldg(reinterpret_cast<const float4*>(s + cv * E + e));
        gg[e] = g4.x; gg[e + 1] = g4.y; gg[e + 2] = g4.z; gg[e + 3] = g4.w;
        ss[e] = s4.x; ss[e + 1] = s4.y; ss[e + 2] = s4.z; ss[e + 3] = s4.w;
      }
      const uint4* X4 = reinterpret_cast<const uint4*>(x) + cv;
      uint4* O4 = reinterpret_cast<uint4*>(out) + cv;
      const long long rstep = gridDim.y;
      for (long long t0 = blockIdx.y; t0 < T_; t0 += kUnroll * rstep) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const long long t = t0 + u * rstep;
          if (t < T_) v[u] = X4[t * vrow];
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const long long t = t0 + u * rstep;
          if (t < T_) {
            float f[E];
            Vec16<T>::unpack(v[u], f);
#pragma unroll
            for (int e = 0; e < E; ++e) f[e] = body_tanh<T>(f[e] * gg[e]) * ss[e];
            O4[t * vrow] = Vec16<T>::pack(f);
          }
        }
      }
    }
  } else {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
      const int c = (int)(i % d);
      store_elem(out + i, body_tanh<T>(load_elem(x + i) * g[c]) * s[c]);
    }
  }
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kEwThreads) synth_layer_backward_kernel(const T* x, const float* __restrict__ g,
                                                                          const float* __restrict__ s, const T* dva,
                                                                          const T* dvb, T* dx, long long T_, int d) {
  pdl_wait();
  pdl_trigger();  // the next kernel may launch once this one's prerequisites are done
  const long long n = T_ * (long long)d;
  const long long stride = (long long)gridDim.x * blockDim.x;
  if constexpr (VEC) {
    // as synth_layer_kernel: one channel vector per thread, down the tokens
    constexpr int E = Vec16<T>::kElems;
    constexpr int kUnroll = 4;
    const int vrow = d / E;
    const int cv = blockIdx.x * blockDim.x + threadIdx.x;
    if (cv < vrow) {
      float gg[E], ss[E];
#pragma unroll
      for (int e = 0; e < E; e += 4) {
        const float4 g4 = __ldg(reinterpret_cast<const float4*>(g + cv * E + e));
        const float4 s4 = __ldg(reinterpret_cast<const float4*>(s + cv * E + e));
        gg[e] = g4.x; gg[e + 1] = g4.y; gg[e + 2] = g4.z; gg[e + 3] = g4.w;
        ss[e] = s4.x; ss[e + 1] = s4.y; ss[e + 2] = s4.z; ss[e + 3] = s4.w;
      }
      const uint4* X4 = reinterpret_cast<const uint4*>(x) + cv;
      const uint4* A4 = reinterpret_cast<const uint4*>(dva) + cv;
      const uint4* B4 = dvb ? reinterpret_cast<const uint4*>(dvb) + cv : nullptr;
      uint4* O4 = reinterpret_cast<uint4*>(dx) + cv;
      const long long rstep = gridDim.y;
      for (long long t0 = blockIdx.y; t0 < T_; t0 += kUnroll * rstep) {
        uint4 xv[kUnroll], av[kUnroll], bv[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const long long t = t0 + u * rstep;
          if (t < T_) {
            xv[u] = X4[t * vrow];
            av[u] = A4[t * vrow];
            if (B4) bv[u] = B4[t * vrow];
          }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const long long t = t0 + u * rstep;
          if (t < T_) {
            float f[E], ga[E];
            Vec16<T>::unpack(xv[u], f);
            Vec16<T>::unpack(av[u], ga);
            if (B4) {
              float gb[E];
              Vec16<T>::unpack(bv[u], gb);
#pragma unroll
              for (int e = 0; e < E; ++e) ga[e] += gb[e];
            }
#pragma unroll
            for (int e = 0; e < E; ++e) f[e] = ga[e] * sech2(f[e] * gg[e]) * gg[e] * ss[e];
            O4[t * vrow] = Vec16<T>::pack(f);
          }
        }
      }
    }
  } else {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
      const int c = (int)(i % d);
      float dv = load_elem(dva + i);
      if (dvb) dv += load_elem(dvb + i);
      store_elem(dx + i, dv * sech2(load_elem(x + i) * g[c]) * g[c] * s[c]);
    }
  }
}

// ---------------------------------------------------------------- launch --

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Grid of the channel-vector kernels: x covers the vrow vectors of a row
// with kColThreads threads per block, y strides over the tokens, sized to
// threads_per_sm on every SM.  The forward body streams fastest with 1024
// threads per SM (each walks more tokens, fewer blocks); its gradient reads
// three rows per token and keeps 2048.
constexpr int kColThreads = 128;

static dim3 col_grid(int vrow, long long T_, int threads_per_sm) {
  DeviceInfo di;
  if (device_info(&di) != cudaSuccess) di.sm_count = 1;
  const int gx = (vrow + kColThreads - 1) / kColThreads;
  long long gy = (long long)di.sm_count * (threads_per_sm / kColThreads) / gx;
  if (gy > T_) gy = T_;
  if (gy > 65535) gy = 65535;
  if (gy < 1) gy = 1;
  return dim3(gx, (unsigned)gy);
}

static int ew_grid(long long work_items) {
  DeviceInfo di;
  if (device_info(&di) != cudaSuccess) di.sm_count = 1;
  const long long cap = (long long)di.sm_count * kEwCtasPerSm;
  long long g = (work_items + kEwThreads - 1) / kEwThreads;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (int)g;
}

template <typename T>
static cudaError_t launch_fold_t(const void* prev, const void* F, void* dst, long long n, cudaStream_t st) {
  constexpr int E = 16 / (int)sizeof(T);
  const bool vec = n % E == 0 && al16(F) && al16(dst) && (!prev || al16(prev));
  const T* P = static_cast<const T*>(prev);
  const T* Fp = static_cast<const T*>(F);
  T* D = static_cast<T*>(dst);
  const cudaError_t e = vec ? launch_kernel(fold_kernel<T, true>, dim3(ew_grid(n / E)), dim3(kEwThreads), 0, st, P, Fp, D, n)
                           : launch_kernel(fold_kernel<T, false>, dim3(ew_grid(n)), dim3(kEwThreads), 0, st, P, Fp, D, n);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_fold(const void* prev, const void* F, void* dst, int64_t n, int dtype, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  return dtype == ATTNRES_BF16 ? launch_fold_t<bf16_t>(prev, F, dst, n, stream)
                               : launch_fold_t<float>(prev, F, dst, n, stream);
}

template <typename T>
static cudaError_t launch_synth_t(const void* x, const float* g, const float* s, void* out, long long T_, int d,
                                  cudaStream_t st) {
  constexpr int E = 16 / (int)sizeof(T);
  const long long n = T_ * (long long)d;
  // the vector path also reads g and s as float4: they must be 16-byte aligned
  const bool vec = d % E == 0 && al16(x) && al16(out) && al16(g) && al16(s);
  const T* X = static_cast<const T*>(x);
  T* O = static_cast<T*>(out);
  const cudaError_t e =
      vec ? launch_kernel(synth_layer_kernel<T, true>, col_grid(d / E, T_, 1024), dim3(kColThreads), 0, st, X, g, s, O, T_, d)
          : launch_kernel(synth_layer_kernel<T, false>, dim3(ew_grid(n)), dim3(kEwThreads), 0, st, X, g, s, O, T_, d);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_synthetic_layer(const void* x, const float* g, const float* s, void* out, int64_t T, int d,
                                   int dtype, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  return dtype == ATTNRES_BF16 ? launch_synth_t<bf16_t>(x, g, s, out, T, d, stream)
                               : launch_synth_t<float>(x, g, s, out, T, d, stream);
}

template <typename T>
static cudaError_t launch_synth_bwd_t(const void* x, const float* g, const float* s, const void* dva,
                                      const void* dvb, void* dx, long long T_, int d, cudaStream_t st) {
  constexpr int E = 16 / (int)sizeof(T);
  const long long n = T_ * (long long)d;
  // the vector path also reads g and s as float4: they must be 16-byte aligned
  const bool vec = d % E == 0 && al16(x) && al16(dva) && (!dvb || al16(dvb)) && al16(dx) && al16(g) && al16(s);
  const T* X = static_cast<const T*>(x);
  const T* A = static_cast<const T*>(dva);
  const T* B = static_cast<const T*>(dvb);
  T* O = static_cast<T*>(dx);
  const cudaError_t e =
      vec ? launch_kernel(synth_layer_backward_kernel<T, true>, col_grid(d / E, T_, 2048), dim3(kColThreads), 0, st, X, g, s,
                          A, B, O, T_, d)
          : launch_kernel(synth_layer_backward_kernel<T, false>, dim3(ew_grid(n)), dim3(kEwThreads), 0, st, X, g, s, A,
                          B, O, T_, d);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_synthetic_layer_backward(const void* x, const float* g, const float* s, const void* dva,
                                            const void* dvb, void* dx, int64_t T, int d, int dtype,
                                            cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  return dtype == ATTNRES_BF16 ? launch_synth_bwd_t<bf16_t>(x, g, s, dva, dvb, dx, T, d, stream)
                               : launch_synth_bwd_t<float>(x, g, s, dva, dvb, dx, T, d, stream);
}

}  // namespace attnres
