// Shared device-side helpers of the GB300 gate-aggregation library.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tango.h"

namespace tg {

// Error word bits (see tg_check_device_error in tango.h).
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrValue = 2u;
constexpr unsigned kKernTango = 1u << 8;
constexpr unsigned kKernWango = 2u << 8;
constexpr unsigned kKernGemm = 3u << 8;
constexpr unsigned kKernModel = 4u << 8;  // embedding lookup
constexpr unsigned kKernBackward = 5u << 8;

// Kernels receive the address of the per-device error word (owned by api.cu) as an
// argument, so that translation units need no relocatable device code.
__device__ __forceinline__ void record_error(unsigned* err, unsigned bits) { atomicOr(err, bits); }

// Storage-type adapters ----------------------------------------------------
template <typename T> struct io;
template <> struct io<float> {
  static __device__ __forceinline__ float ld(const float* p) { return *p; }
  static __device__ __forceinline__ void st(float* p, float x) { *p = x; }
};
template <> struct io<__nv_bfloat16> {
  static __device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ void st(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
};

// Per-head temperature: the device array if given, else the scalar; clamped to
// the eq. 4 range [0, 20] with an error flag when a device value is outside it.
__device__ __forceinline__ float head_tau(const float* tau, float s, int a, unsigned* err,
                                         unsigned kern) {
  if (!tau) return s;
  float t = tau[a];
  if (!(t >= 0.f && t <= 20.f)) {  // also catches NaN
    record_error(err, kErrValue | kern);
    t = (t > 20.f) ? 20.f : 0.f;
  }
  return t;
}

// log2(e), used to evaluate exp(x) as exp2(x * log2(e)).
constexpr float kLog2e = 1.4426950408889634f;

__host__ __device__ constexpr int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

}  // namespace tg
