// actfn.cuh -- activation functions and their derivatives in fp32, plus bf16 packing.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"

namespace dm {

// Logistic sigmoid through the hardware exponential and approximate division intrinsics
// (relative error ~1e-6, far below the bf16 rounding of every value it feeds).  For large -x the
// exponential overflows to +inf and the quotient is 0, the correct limit.
__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// GeLU in its exact form x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)).
__device__ __forceinline__ float act_fwd(int act, float x) {
  if (act == ACT_RELU) return fmaxf(x, 0.0f);
  if (act == ACT_GELU) return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
  return x;
}

// d act / dz.  GeLU: Phi(z) + z phi(z).
__device__ __forceinline__ float act_grad(int act, float z) {
  if (act == ACT_RELU) return z > 0.0f ? 1.0f : 0.0f;
  if (act == ACT_GELU) {
    const float cdf = 0.5f * (1.0f + erff(z * 0.70710678118654752f));
    const float pdf = 0.39894228040143268f * expf(-0.5f * z * z);
    return cdf + z * pdf;
  }
  return 1.0f;
}

// Gated: SwiGLU silu(g) * u, bilinear g * u.
__device__ __forceinline__ float glu_fwd(int act, float g, float u) {
  if (act == ACT_SWIGLU) return g * sigmoidf_(g) * u;
  return g * u;
}

__device__ __forceinline__ void glu_bwd(int act, float g, float u, float dh, float& dg, float& du,
                                        float& hv) {
  if (act == ACT_SWIGLU) {
    const float s = sigmoidf_(g);
    const float silu = g * s;
    hv = silu * u;
    du = dh * silu;
    dg = dh * u * s * (1.0f + g * (1.0f - s));
  } else {
    hv = g * u;
    du = dh * g;
    dg = dh * u;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace dm
