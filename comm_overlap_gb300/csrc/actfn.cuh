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

// Standard normal CDF Phi(x) and density phi(x) with one exponential.  Phi(x) = (1 + erf(u)) / 2,
// u = x / sqrt 2, with erf from Abramowitz & Stegun, Handbook of Mathematical Functions, formula
// 7.1.26: erf(u) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-u^2), t = 1 / (1 + p u), for
// u >= 0 (|error| <= 1.5e-7), odd extension for u < 0.  exp(-u^2) = exp(-x^2 / 2) is also the
// unnormalised density, so phi comes for free.
__device__ __forceinline__ void normal_cdf_pdf(float x, float& cdf, float& pdf) {
  const float u = fabsf(x) * 0.70710678118654752f;
  const float t = __fdividef(1.0f, fmaf(0.3275911f, u, 1.0f));
  const float poly =
      t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f), -0.284496736f), 0.254829592f);
  const float e = __expf(-0.5f * x * x);
  const float erf_abs = 1.0f - poly * e;  // erf(|u|)
  cdf = 0.5f + copysignf(0.5f * erf_abs, x);
  pdf = 0.39894228040143268f * e;
}

// GeLU in its exact form x * Phi(x) (Phi through normal_cdf_pdf).
__device__ __forceinline__ float act_fwd(int act, float x) {
  if (act == ACT_RELU) return fmaxf(x, 0.0f);
  if (act == ACT_GELU) {
    float cdf, pdf;
    normal_cdf_pdf(x, cdf, pdf);
    return x * cdf;
  }
  return x;
}

// d act / dz.  GeLU: Phi(z) + z phi(z).
__device__ __forceinline__ float act_grad(int act, float z) {
  if (act == ACT_RELU) return z > 0.0f ? 1.0f : 0.0f;
  if (act == ACT_GELU) {
    float cdf, pdf;
    normal_cdf_pdf(z, cdf, pdf);
    return fmaf(z, pdf, cdf);
  }
  return 1.0f;
}

// act(z) and act'(z) together (one CDF/density evaluation for GeLU).
__device__ __forceinline__ void act_fwd_grad(int act, float z, float& h, float& d) {
  if (act == ACT_GELU) {
    float cdf, pdf;
    normal_cdf_pdf(z, cdf, pdf);
    h = z * cdf;
    d = fmaf(z, pdf, cdf);
  } else if (act == ACT_RELU) {
    h = fmaxf(z, 0.0f);
    d = z > 0.0f ? 1.0f : 0.0f;
  } else {
    h = z;
    d = 1.0f;
  }
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
