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
// RoPE rotation for pair k at position pos: angle = pos * base^(-2k/d_r).
// The frequencies are computed once on the host in double precision and handed to the
// kernels as float pairs (f = hi + lo). The angle is formed in float-float arithmetic and
// reduced modulo 2 pi by the Cody-Waite method (two-term 2 pi, fused multiply-adds), so that
// long contexts keep float accuracy in the rotation without any double arithmetic on the
// device. Positions are split into a multiple of 4096 and a remainder, both exact in float.
// ----------------------------------------------------------------------------------
constexpr int kMaxRopePairs = 64;  // d_h^R <= 128

struct RopeFreqs {
  float hi[kMaxRopePairs];
  float lo[kMaxRopePairs];
};

inline RopeFreqs rope_freqs(const mla_dims_t* d) {
  RopeFreqs f{};
  for (int k = 0; k < d->d_hr / 2 && k < kMaxRopePairs; ++k) {
    const double v = pow((double)d->rope_base, -2.0 * (double)k / (double)d->d_hr);
    f.hi[k] = (float)v;
    f.lo[k] = (float)(v - (double)f.hi[k]);
  }
  return f;
}

// pos * (fh + fl) reduced into [-pi, pi] (a few float ulps of pi)
__device__ __forceinline__ float rope_reduce(float pos_part, float fh, float fl) {
  constexpr float kInv2Pi = 0.15915494309189535f;
  constexpr float k2PiHi = 6.28318548202514648f;     // float nearest to 2 pi
  constexpr float k2PiLo = -1.7484556000744883e-7f;  // 2 pi - k2PiHi
  const float a_hi = pos_part * fh;
  const float a_lo = fmaf(pos_part, fh, -a_hi) + pos_part * fl;
  const float n = rintf(a_hi * kInv2Pi);
  float r = fmaf(-n, k2PiHi, a_hi);
  r = fmaf(-n, k2PiLo, r);
  return r + a_lo;
}

// cos and sin of pos * (fh + fl)
__device__ __forceinline__ void rope_cs_f(int pos, float fh, float fl, float* c, float* s) {
  const float r = rope_reduce((float)(pos & ~4095), fh, fl) + rope_reduce((float)(pos & 4095), fh, fl);
  sincosf(r, s, c);
}

__device__ __forceinline__ void rope_cs(int pos, int k, const RopeFreqs& f, float* c, float* s) {
  rope_cs_f(pos, f.hi[k], f.lo[k], c, s);
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
