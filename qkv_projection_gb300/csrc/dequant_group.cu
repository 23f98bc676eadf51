// Per-group dequantisation and its straight-through backward, elementwise
// over [outer, axis] with one scale per group of `group` consecutive elements
// of the last axis.
//
// What they compute ("baracuda-kernels -- src/quantize/dequantize_per_group_
// backward.rs", module doc and DequantizePerGroupBackwardPlan doc):
//   backward  dx[i, j]  = dy[i, j] * scale[i, j / group]      (T = f32, f64, f16, bf16)
//   forward   out[i, j] = T(q[i, j]) * scale[i, j / group]    (q int8 or uint8)
// Each product is rounded once to T: for f16 and bf16 operands it is exact in
// f32, so it is formed in f32 and rounded once (deterministic, bit-stable).
//
// Both are HBM-bound streams: every thread moves 16-byte vectors of the output
// (and the matching bytes of the input) with L1-bypassing loads and streaming
// stores, several vectors in flight per thread; the scale row is read through
// the cache (each scale serves group / vector-length threads).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "kaio_internal.h"

namespace kaio {
namespace {

template <typename T> struct Elt;
template <> struct Elt<float> {
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elt<__half> {
  static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
  static __device__ __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
};
template <> struct Elt<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// One product, rounded once to T. f64 multiplies in f64; f32 in f32; f16 and
// bf16 in f32, where the product of two such values (or of an 8-bit integer and
// one) is exact, then round once.
template <typename T, typename A>
__device__ __forceinline__ T scaled(A a, T s) {
  if constexpr (sizeof(T) == 8) {
    return static_cast<double>(a) * s;
  } else {
    float af;
    if constexpr (sizeof(A) == 1) af = static_cast<float>(a);
    else af = Elt<T>::to_f(a);
    return Elt<T>::from_f(af * Elt<T>::to_f(s));
  }
}

// A: input element (T for the backward, int8/uint8 for the forward).
// VEC elements per vector = 16 bytes of output.
template <typename T, typename A>
struct Vec {
  static constexpr int kN = 16 / static_cast<int>(sizeof(T));
  static constexpr int kInBytes = kN * static_cast<int>(sizeof(A));
};

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream4(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint16_t ld_stream2(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream16(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Input bytes of one vector, as an array of kN elements of A.
template <typename T, typename A>
struct InVec {
  static constexpr int kN = Vec<T, A>::kN;
  A e[kN];
  __device__ __forceinline__ void load(const A* p) {
    constexpr int b = Vec<T, A>::kInBytes;
    if constexpr (b == 16) {
      const uint4 v = ld_stream16(p);
      memcpy(e, &v, 16);
    } else if constexpr (b == 8) {
      const uint2 v = ld_stream8(p);
      memcpy(e, &v, 8);
    } else if constexpr (b == 4) {
      const uint32_t v = ld_stream4(p);
      memcpy(e, &v, 4);
    } else {
      static_assert(b == 2, "input vector of 2, 4, 8 or 16 bytes");
      const uint16_t v = ld_stream2(p);
      memcpy(e, &v, 2);
    }
  }
};

constexpr int kThreads = 256;
constexpr int kUnroll = 4;   // vectors in flight per thread

// Vector kernel: requires axis % kN == 0 and 16-byte (output) / kInBytes
// (input) aligned pointers. kOneGroup: group % kN == 0, so a vector lies in
// one group and needs one scale.
template <typename T, typename A, bool kOneGroup>
__global__ void __launch_bounds__(kThreads)
    dequant_group_vec_kernel(const A* __restrict__ in, const T* __restrict__ scale, T* __restrict__ out,
                             long long nvec, int axis, int group, int ngroups) {
  constexpr int kN = Vec<T, A>::kN;
  const int vpr = axis / kN;                              // vectors per row
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long v0 = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; v0 < nvec;
       v0 += stride * kUnroll) {
    InVec<T, A> x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long v = v0 + u * stride;
      if (v < nvec) x[u].load(in + v * kN);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long v = v0 + u * stride;
      if (v >= nvec) continue;
      const long long row = v / vpr;
      const int j = static_cast<int>(v - row * vpr) * kN;
      const T* srow = scale + row * ngroups;
      T r[kN];
      if (kOneGroup) {
        const T s = __ldg(srow + j / group);
#pragma unroll
        for (int t = 0; t < kN; ++t) r[t] = scaled<T>(x[u].e[t], s);
      } else {
#pragma unroll
        for (int t = 0; t < kN; ++t) r[t] = scaled<T>(x[u].e[t], __ldg(srow + (j + t) / group));
      }
      uint4 o;
      memcpy(&o, r, 16);
      st_stream16(out + v * kN, o);
    }
  }
}

// Any shape and alignment: one element per thread per step.
template <typename T, typename A>
__global__ void __launch_bounds__(kThreads)
    dequant_group_scalar_kernel(const A* __restrict__ in, const T* __restrict__ scale, T* __restrict__ out,
                                long long total, int axis, int group, int ngroups) {
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long e = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; e < total; e += stride) {
    const long long row = e / axis;
    const int j = static_cast<int>(e - row * axis);
    out[e] = scaled<T>(in[e], __ldg(scale + row * ngroups + j / group));
  }
}

template <typename T, typename A>
cudaError_t launch_typed(const void* in_, const void* scale_, void* out_, int outer, int axis, int group,
                         int num_sms, cudaStream_t stream) {
  const A* in = static_cast<const A*>(in_);
  const T* scale = static_cast<const T*>(scale_);
  T* out = static_cast<T*>(out_);
  constexpr int kN = Vec<T, A>::kN;
  const long long total = static_cast<long long>(outer) * axis;
  const int ngroups = axis / group;
  const bool aligned = reinterpret_cast<uintptr_t>(out) % 16 == 0 &&
                       reinterpret_cast<uintptr_t>(in) % Vec<T, A>::kInBytes == 0;
  // One pass per thread (kUnroll vectors) where the grid allows: short-lived
  // CTAs that the block scheduler refills measured faster on these streams
  // than a persistent grid-stride grid (a ragged last wave of resident CTAs
  // leaves HBM idle). Very large problems stride over the capped grid.
  const int max_blocks = num_sms * 64;
  if (aligned && axis % kN == 0) {
    const long long nvec = total / kN;
    const long long want = (nvec + kThreads * kUnroll - 1) / (kThreads * kUnroll);
    const int blocks = static_cast<int>(want < max_blocks ? (want < 1 ? 1 : want) : max_blocks);
    if (group % kN == 0)
      dequant_group_vec_kernel<T, A, true><<<blocks, kThreads, 0, stream>>>(in, scale, out, nvec, axis, group, ngroups);
    else
      dequant_group_vec_kernel<T, A, false><<<blocks, kThreads, 0, stream>>>(in, scale, out, nvec, axis, group, ngroups);
  } else {
    const long long want = (total + kThreads - 1) / kThreads;
    const int blocks = static_cast<int>(want < max_blocks ? want : max_blocks);
    dequant_group_scalar_kernel<T, A><<<blocks, kThreads, 0, stream>>>(in, scale, out, total, axis, group, ngroups);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dequant_group_backward(FloatType t, const void* dy, const void* scale, void* dx,
                                          int outer, int axis, int group, int num_sms, cudaStream_t stream) {
  switch (t) {
    case FloatType::F32: return launch_typed<float, float>(dy, scale, dx, outer, axis, group, num_sms, stream);
    case FloatType::F64: return launch_typed<double, double>(dy, scale, dx, outer, axis, group, num_sms, stream);
    case FloatType::F16: return launch_typed<__half, __half>(dy, scale, dx, outer, axis, group, num_sms, stream);
    case FloatType::BF16:
      return launch_typed<__nv_bfloat16, __nv_bfloat16>(dy, scale, dx, outer, axis, group, num_sms, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_dequant_group_forward(FloatType t, bool q_unsigned, const void* q, const void* scale,
                                         void* out, int outer, int axis, int group, int num_sms,
                                         cudaStream_t stream) {
#define KAIO_FWD(TT)                                                                                 \
  return q_unsigned ? launch_typed<TT, uint8_t>(q, scale, out, outer, axis, group, num_sms, stream) \
                    : launch_typed<TT, int8_t>(q, scale, out, outer, axis, group, num_sms, stream)
  switch (t) {
    case FloatType::F32: KAIO_FWD(float);
    case FloatType::F64: KAIO_FWD(double);
    case FloatType::F16: KAIO_FWD(__half);
    case FloatType::BF16: KAIO_FWD(__nv_bfloat16);
  }
#undef KAIO_FWD
  return cudaErrorInvalidValue;
}

}  // namespace kaio
