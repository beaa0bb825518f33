/*
 * oracle.c -- CPU oracle for the chunked tensor-parallel MLP.  TEST INFRASTRUCTURE ONLY:
 * loaded by the test suite, the smoke check and the benchmark's CPU-baseline leg, never by
 * the product path.  Plain C, double-precision arithmetic, OpenMP over independent rows or
 * features.  See oracle.h for the definitions and the passages they follow.
 */
#include "oracle.h"

#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_NONE = 0, ORC_RELU = 1, ORC_GELU = 2, ORC_SWIGLU = 3, ORC_BILINEAR = 4 };

static inline double bf16_bits_to_double(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* ---- elementwise functions ----------------------------------------------------------- */

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* GeLU in its exact form x * Phi(x), Phi the standard normal CDF (the pages say only
 * "GeLU"; the erf form is the definition, the tanh form an approximation of it). */
double oracle_act(int act, double z) {
  switch (act) {
    case ORC_RELU: return z > 0.0 ? z : 0.0;
    case ORC_GELU: return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));
    default: return z;
  }
}

double oracle_act_grad(int act, double z) {
  switch (act) {
    case ORC_RELU: return z > 0.0 ? 1.0 : 0.0;
    case ORC_GELU: {
      const double cdf = 0.5 * (1.0 + erf(z / sqrt(2.0)));
      const double pdf = exp(-0.5 * z * z) / sqrt(2.0 * M_PI);
      return cdf + z * pdf;
    }
    default: return 1.0;
  }
}

/* SwiGLU: silu(gate) * up, silu(g) = g * sigmoid(g).  Bilinear: gate * up. */
double oracle_glu(int act, double g, double u) {
  if (act == ORC_SWIGLU) return g * sigmoid(g) * u;
  return g * u;
}

double oracle_glu_dg(int act, double g, double u) {
  if (act == ORC_SWIGLU) {
    const double s = sigmoid(g);
    return u * s * (1.0 + g * (1.0 - s));
  }
  return u;
}

double oracle_glu_du(int act, double g, double u) {
  (void)u;
  if (act == ORC_SWIGLU) return g * sigmoid(g);
  return g;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---- instantiations of the arithmetic ------------------------------------------------ */

#define LD_BF16(p, i) bf16_bits_to_double((p)[i])
#define LD_F64(p, i) ((double)(p)[i])

/* bf16 activations, bf16 weights: the public entry points */
#define SFX bf16
#define AT uint16_t
#define ALD LD_BF16
#define WT uint16_t
#define WLD LD_BF16
#include "oracle_core.inc"
#undef SFX
#undef AT
#undef ALD
#undef WT
#undef WLD

/* double activations and weights: for finite-difference checks */
#define SFX f64
#define AT double
#define ALD LD_F64
#define WT double
#define WLD LD_F64
#include "oracle_core.inc"
#undef SFX
#undef AT
#undef ALD
#undef WT
#undef WLD

/* double activations, bf16 weights: the layer stack, whose activations stay in double */
#define SFX mix
#define AT double
#define ALD LD_F64
#define WT uint16_t
#define WLD LD_BF16
#include "oracle_core.inc"
#undef SFX
#undef AT
#undef ALD
#undef WT
#undef WLD

/* Pre-LN residual stack ([Domino] "实现与优化": LayerNorm and residual between sublayers;
 * forward schedule of figure 9).  Each row is independent through LN, the MLP and the
 * residual, so rows are evaluated one at a time in double, with no intermediate rounding. */
int oracle_stack_fwd_bf16(int L, int64_t M, int64_t h, int64_t F, int t, int act, double eps,
                          const uint16_t* Z0, const uint16_t* A, const uint16_t* B,
                          const int64_t* rows, int64_t n_rows, double* Zout) {
  if (L < 0 || M < 0 || h <= 0 || F <= 0 || t <= 0 || F % t != 0 || act < 0 || act > ORC_BILINEAR)
    return -1;
  const int gated = (act == ORC_SWIGLU || act == ORC_BILINEAR);
  const int64_t a_layer = (gated ? 2 * F : F) * h, b_layer = h * F;
  const int64_t n = rows ? n_rows : M;
  int bad = 0;
#pragma omp parallel
  {
    double* work = (double*)malloc(sizeof(double) * (size_t)(4 * F + 3 * h));
    double* Hrow = work + 3 * F;
    double* z = work + 4 * F;
    double* ln = z + h;
    double* y = ln + h;
#pragma omp for schedule(dynamic, 1)
    for (int64_t rr = 0; rr < n; ++rr) {
      const int64_t r = rows ? rows[rr] : rr;
      if (r < 0 || r >= M) { bad = 1; continue; }
      for (int64_t k = 0; k < h; ++k) z[k] = bf16_bits_to_double(Z0[r * h + k]);
      for (int l = 0; l < L; ++l) {
        layernorm_rowmix(h, eps, z, ln);
        fwd_rowmix(h, F, t, act, ln, A + l * a_layer, B + l * b_layer, 0, Hrow, y, work);
        for (int64_t k = 0; k < h; ++k) z[k] += y[k];
      }
      for (int64_t k = 0; k < h; ++k) Zout[rr * h + k] = z[k];
    }
    free(work);
  }
  return bad ? -2 : 0;
}
