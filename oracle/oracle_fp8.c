/*
 * oracle_fp8.c -- CPU oracle for the FP8 variant of the MLP forward.  TEST INFRASTRUCTURE ONLY:
 * loaded by the test suite, the smoke check and the benchmark's CPU-baseline leg, never by the
 * product path.  Plain C, double precision, OpenMP over independent rows.
 *
 * "04 · TP/SP 的通信-计算 overlap 与工程优化", section 4 (与其它并行的 overlap 耦合, on FP8): the
 * activations can be moved in FP8 to halve the bandwidth, but the reduction of partial sums must
 * accumulate in higher precision.  The variant computed here: the GEMM operands in FP8 E4M3 with
 * per-tensor scales, the first-linear output re-quantised to E4M3 for the second linear, and the
 * shard partials and their sum kept in higher precision:
 *
 *   Z = sx sa (X8 . A8^T)           (real values: X = sx X8, A = sa A8, codes decoded exactly)
 *   H = act(Z)  (gated: glu(G, U))
 *   H8 = e4m3(H / sh), the quotient rounded to fp32 first (the precision in which the GPU takes
 *        the same decision), then to the nearest E4M3 value, ties to even, saturating at +-448
 *   Y = sh sb (H8 . B8^T)           (sum over every shard's columns, i.e. the reduced partials)
 *
 * E4M3 (OCP 8-bit floating point, E4M3 variant): sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; exponent 0 holds the subnormals m 2^-9; no infinities; S.1111.111 is NaN; the largest
 * finite magnitude is 1.75 2^8 = 448.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

double oracle_e4m3_decode(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

/* Nearest E4M3 value of x (an fp32 value held in a double), ties to even, saturating. */
uint8_t oracle_e4m3_encode(double x) {
  if (isnan(x)) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  if (a >= 464.0) return sign | 0x7E; /* at or past the midpoint 448 / 480 (480 is not finite) */
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: steps of 2^-9; 8 steps is the smallest normal 2^-6 (code 0x08) */
    const double q = rint(a * 512.0); /* exact scaling by 2^9; rint rounds half to even */
    return sign | (uint8_t)q;
  }
  int e2;
  frexp(a, &e2);            /* a = f 2^e2, f in [0.5, 1): the leading bit is 2^(e2-1) */
  const int e = e2 - 1;     /* a in [2^e, 2^(e+1)) */
  double q = rint(ldexp(a, 3 - e)); /* in [8, 16], steps of 2^(e-3) */
  int ee = e;
  if (q == 16.0) {
    q = 8.0;
    ++ee;
  }
  const int code = ((ee + 7) << 3) | ((int)q - 8);
  return sign | (uint8_t)code;
}

int oracle_mlp_fwd_fp8(int64_t M, int64_t h, int64_t F, int t, int act, const uint8_t* X8, const uint8_t* A8,
                       const uint8_t* B8, double sx, double sa, double sb, double sh, const int64_t* rows,
                       int64_t n_rows, double* Y, uint8_t* H8_out) {
  if (M < 0 || h <= 0 || F <= 0 || t <= 0 || F % t != 0 || act < 0 || act > 4 || !(sh > 0.0)) return -1;
  const int gated = (act == 3 || act == 4);
  const int64_t Fi = F / t;
  const int64_t n = rows ? n_rows : M;
  double dec[256];
  for (int c = 0; c < 256; ++c) dec[c] = oracle_e4m3_decode((uint8_t)c);
  int bad = 0;
#pragma omp parallel
  {
    double* x = (double*)malloc(sizeof(double) * (size_t)(h + F));
    double* hq = x + h; /* decoded H8 of the row */
#pragma omp for schedule(dynamic, 1)
    for (int64_t rr = 0; rr < n; ++rr) {
      const int64_t r = rows ? rows[rr] : rr;
      if (r < 0 || r >= M) {
        bad = 1;
        continue;
      }
      for (int64_t k = 0; k < h; ++k) x[k] = dec[X8[r * h + k]];
      for (int64_t f = 0; f < F; ++f) {
        const int64_t i = f / Fi, j = f % Fi;
        double hv;
        if (gated) {
          double g = 0.0, u = 0.0;
          const uint8_t* ag = A8 + (i * 2 * Fi + j) * h;
          const uint8_t* au = A8 + (i * 2 * Fi + Fi + j) * h;
          for (int64_t k = 0; k < h; ++k) {
            g += x[k] * dec[ag[k]];
            u += x[k] * dec[au[k]];
          }
          hv = oracle_glu(act, sx * sa * g, sx * sa * u);
        } else {
          double z = 0.0;
          const uint8_t* af = A8 + f * h;
          for (int64_t k = 0; k < h; ++k) z += x[k] * dec[af[k]];
          hv = oracle_act(act, sx * sa * z);
        }
        const uint8_t code = oracle_e4m3_encode((double)(float)(hv / sh));
        hq[f] = dec[code];
        if (H8_out) H8_out[rr * F + f] = code;
      }
      for (int64_t c = 0; c < h; ++c) {
        double s = 0.0;
        for (int64_t f = 0; f < F; ++f) s += hq[f] * dec[B8[(f / Fi) * h * Fi + c * Fi + (f % Fi)]];
        Y[rr * h + c] = sh * sb * s;
      }
    }
    free(x);
  }
  return bad ? -2 : 0;
}
