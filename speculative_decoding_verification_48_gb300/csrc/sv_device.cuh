// Device helpers shared by the verification kernels: element types, PTX
// helpers and warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <type_traits>

#include "sv_internal.h"

namespace sv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTinyT = 1e-20f;
// Bound of every device-side wait, in SM clock cycles (about one second at
// 2 GHz).
constexpr long long kWaitCycles = 2000000000LL;

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max that returns NaN when either input is NaN
__device__ __forceinline__ float max_nan(float a, float b) {
  float y;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

// ---------------------------------------------------------------------------
// Element types
// ---------------------------------------------------------------------------

template <int DT> struct Elt;

template <> struct Elt<SV_F32> {
  using T = float;
  static constexpr int kVec = 4;
  __device__ static __forceinline__ void unpack(const uint4 &r, float *o) {
    o[0] = __uint_as_float(r.x); o[1] = __uint_as_float(r.y);
    o[2] = __uint_as_float(r.z); o[3] = __uint_as_float(r.w);
  }
  __device__ static __forceinline__ float load1(const T *p) { return __ldg(p); }
};

template <> struct Elt<SV_BF16> {
  using T = __nv_bfloat16;
  static constexpr int kVec = 8;
  // bf16 -> f32 is a 16-bit left shift of the bit pattern (exact).
  __device__ static __forceinline__ void unpack(const uint4 &r, float *o) {
    const unsigned w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static __forceinline__ void unpack(const uint2 &r, float *o) {
    o[0] = __uint_as_float(r.x << 16); o[1] = __uint_as_float(r.x & 0xffff0000u);
    o[2] = __uint_as_float(r.y << 16); o[3] = __uint_as_float(r.y & 0xffff0000u);
  }
  __device__ static __forceinline__ float load1(const T *p) {
    const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(p));
    return __uint_as_float(static_cast<unsigned>(b) << 16);
  }
};

template <> struct Elt<SV_F16> {
  using T = __half;
  static constexpr int kVec = 8;
  __device__ static __forceinline__ void unpack(const uint4 &r, float *o) {
    const unsigned w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
      float2 f = __half22float2(h);
      o[2 * i] = f.x;
      o[2 * i + 1] = f.y;
    }
  }
  __device__ static __forceinline__ void unpack(const uint2 &r, float *o) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
  }
  __device__ static __forceinline__ float load1(const T *p) {
    const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(p));
    return __half2float(__ushort_as_half(b));
  }
};

// ---------------------------------------------------------------------------
// Warp reductions
// ---------------------------------------------------------------------------

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }
__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_max_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// A temperature the verification cannot use: NaN, or positive but so small
// that l / T overflows.
__device__ __forceinline__ bool bad_temperature(float T) {
  return isnan(T) || (T > 0.f && T < kTinyT);
}

}  // namespace sv
