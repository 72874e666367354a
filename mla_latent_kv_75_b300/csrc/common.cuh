// Shared device/host helpers of libmla (no MLA arithmetic lives here beyond RoPE angles).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

// ----------------------------------------------------------------------------------
// Device status word: the first kernel-detected problem is latched here (0 = none).
// ----------------------------------------------------------------------------------
extern __device__ unsigned int g_status;

__device__ __forceinline__ void flag_status(unsigned int code) {
  atomicCAS(&g_status, 0u, code);
}

// ----------------------------------------------------------------------------------
// Element conversion
// ----------------------------------------------------------------------------------
template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <> __device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }

// ----------------------------------------------------------------------------------
// RoPE angle: pos * base^(-2k/d_r), reduced modulo 2*pi in double precision so that long
// contexts (positions up to 2^31) keep full float accuracy in the rotation.
// ----------------------------------------------------------------------------------
__device__ __forceinline__ void rope_cs(int pos, int k, int d_r, float base, float* c, float* s) {
  const double theta = pow((double)base, -2.0 * (double)k / (double)d_r);
  const double two_pi = 6.283185307179586476925286766559;
  double a = (double)pos * theta;
  a = a - two_pi * floor(a / two_pi);
  sincosf((float)a, s, c);
}

// ----------------------------------------------------------------------------------
// Host helpers
// ----------------------------------------------------------------------------------
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline mla_status_t launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

inline size_t elem_bytes(const mla_dims_t* d) { return d->dtype == MLA_BF16 ? 2 : 4; }

inline float softmax_scale(const mla_dims_t* d) {
  return d->scale != 0.f ? d->scale : 1.0f / sqrtf((float)(d->d_hc + d->d_hr));
}

}  // namespace mla
