/*
 * oracle_attn.c -- CPU oracle for the attention sublayer and the full transformer block of the
 * tensor-parallel layer.  TEST INFRASTRUCTURE ONLY: loaded by the test suite, the smoke check
 * and the benchmark's CPU-baseline leg, never by the product path.  Plain C, double-precision
 * arithmetic from the exact values of the bf16 inputs; OpenMP over independent rows.
 *
 * [Domino] "DeepSpeed-Domino 深度解析…", section "TP 的数据依赖：通信为何难以隐藏": a layer is
 * XAB=Y followed by AllReduce(Y); for the attention layer X is the input, A the attention
 * computation (multi-head attention) and B a linear layer.  Section "实现与优化", figure 9: a
 * Transformer block is one self-attention layer and one MLP layer, with LayerNorm and residual
 * between them.  Tensor parallelism splits the attention by heads (Megatron style): shard i owns
 * heads i*nh_i .. (i+1)*nh_i - 1, nh_i = heads / t, computes their attention and its partial of
 * the output projection; the AllReduce sums the partials.
 *
 * Definitions (d = h / heads, causal self-attention within each sequence of `seq` tokens; token
 * r is position r % seq of sequence r / seq):
 *   q_r = x_r . Wq[head]^T,  k_p = x_p . Wk[head]^T,  v_p = x_p . Wv[head]^T   (d each)
 *   o_r[head] = sum_{p <= pos(r)} w_p v_p,  w = softmax_p(q_r . k_p / sqrt(d)) over p <= pos(r)
 *   y_r = sum_head o_r[head] . Wo[:, head]^T
 * Storage (row-major, nn.Linear [out, in]):
 *   X: M x h.  Wqkv: t shards, shard i is (3 nh_i d) x h: its nh_i query heads (d rows each),
 *   then its key heads, then its value heads.  Wo: t shards, shard i is h x (nh_i d); column
 *   j*d + e of shard i multiplies element e of the shard's local head j.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static inline double bf(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Row of the projection of x (h doubles) by the weight row `w` (h bf16). */
static double dot_w(int64_t h, const double* x, const uint16_t* w) {
  double s = 0.0;
  for (int64_t k = 0; k < h; ++k) s += x[k] * bf(w[k]);
  return s;
}

/* Query, key and value of every head for one token (each heads*d, global head order). */
static void qkv_row(int64_t h, int heads, int t, const double* x, const uint16_t* Wqkv, double* q, double* k,
                    double* v) {
  const int64_t d = h / heads, nhi = heads / t, rows_i = 3 * nhi * d;
  for (int hd = 0; hd < heads; ++hd) {
    const int64_t i = hd / nhi, j = hd % nhi;
    const uint16_t* Wi = Wqkv + i * rows_i * h;
    for (int64_t e = 0; e < d; ++e) {
      q[hd * d + e] = dot_w(h, x, Wi + (0 * nhi * d + j * d + e) * h);
      k[hd * d + e] = dot_w(h, x, Wi + (1 * nhi * d + j * d + e) * h);
      v[hd * d + e] = dot_w(h, x, Wi + (2 * nhi * d + j * d + e) * h);
    }
  }
}

/* Attention output of one query position `pos` over keys/values of positions 0..pos (each row
 * heads*d), into o (heads*d); w: pos+1 doubles of scratch. */
static void attend(int heads, int64_t d, int64_t pos, const double* q, const double* K, const double* V,
                   double* o, double* w) {
  const double scale = 1.0 / sqrt((double)d);
  for (int hd = 0; hd < heads; ++hd) {
    double mx = -INFINITY;
    for (int64_t p = 0; p <= pos; ++p) {
      double s = 0.0;
      for (int64_t e = 0; e < d; ++e) s += q[hd * d + e] * K[p * heads * d + hd * d + e];
      w[p] = s * scale;
      if (w[p] > mx) mx = w[p];
    }
    double sum = 0.0;
    for (int64_t p = 0; p <= pos; ++p) {
      w[p] = exp(w[p] - mx);
      sum += w[p];
    }
    for (int64_t e = 0; e < d; ++e) {
      double acc = 0.0;
      for (int64_t p = 0; p <= pos; ++p) acc += w[p] * V[p * heads * d + hd * d + e];
      o[hd * d + e] = acc / sum;
    }
  }
}

/* Output projection of one token: y = sum over heads of o . Wo^T.  sharded = 0: one sum over the
 * unsharded column index; sharded = 1: shard i's partial over its heads, then the partials
 * summed in shard order 0..t-1 (the reduction the AllReduce performs). */
static void out_proj(int64_t h, int heads, int t, int sharded, const double* o, const uint16_t* Wo, double* y) {
  const int64_t d = h / heads, nhi = heads / t, cols_i = nhi * d;
  for (int64_t c = 0; c < h; ++c) {
    if (!sharded) {
      double s = 0.0;
      for (int64_t col = 0; col < heads * d; ++col) {
        const int64_t i = col / cols_i, jj = col % cols_i;
        s += o[col] * bf(Wo[i * h * cols_i + c * cols_i + jj]);
      }
      y[c] = s;
    } else {
      double tot = 0.0;
      for (int i = 0; i < t; ++i) {
        double p = 0.0;
        for (int64_t jj = 0; jj < cols_i; ++jj) p += o[i * cols_i + jj] * bf(Wo[i * h * cols_i + c * cols_i + jj]);
        tot += p;
      }
      y[c] = tot;
    }
  }
}

static int attn_shape_ok(int64_t M, int64_t h, int heads, int64_t seq, int t) {
  return M >= 0 && h > 0 && heads > 0 && t > 0 && seq > 0 && h % heads == 0 && heads % t == 0 && M % seq == 0;
}

int oracle_attn_fwd_bf16(int64_t M, int64_t h, int heads, int64_t seq, int t, const uint16_t* X,
                         const uint16_t* Wqkv, const uint16_t* Wo, const int64_t* rows, int64_t n_rows, int sharded,
                         double* Y) {
  if (!attn_shape_ok(M, h, heads, seq, t)) return -1;
  const int64_t d = h / heads, hd_all = heads * d;
  const int64_t n = rows ? n_rows : M;
  for (int64_t rr = 0; rr < n; ++rr) {
    const int64_t r = rows ? rows[rr] : rr;
    if (r < 0 || r >= M) return -2;
  }
  /* keys and values of every position up to the row, computed per requested row (rows are
   * independent; for a full evaluation the rows of one sequence share them below) */
  if (!rows) {
    const int64_t nseq = M / seq;
    for (int64_t sq = 0; sq < nseq; ++sq) {
      double* K = (double*)malloc(sizeof(double) * (size_t)(seq * hd_all));
      double* V = (double*)malloc(sizeof(double) * (size_t)(seq * hd_all));
      double* Q = (double*)malloc(sizeof(double) * (size_t)(seq * hd_all));
#pragma omp parallel
      {
        double* x = (double*)malloc(sizeof(double) * (size_t)h);
#pragma omp for schedule(static)
        for (int64_t p = 0; p < seq; ++p) {
          for (int64_t k = 0; k < h; ++k) x[k] = bf(X[(sq * seq + p) * h + k]);
          qkv_row(h, heads, t, x, Wqkv, Q + p * hd_all, K + p * hd_all, V + p * hd_all);
        }
        free(x);
      }
#pragma omp parallel
      {
        double* o = (double*)malloc(sizeof(double) * (size_t)(hd_all + seq));
        double* w = o + hd_all;
#pragma omp for schedule(dynamic, 1)
        for (int64_t p = 0; p < seq; ++p) {
          attend(heads, d, p, Q + p * hd_all, K, V, o, w);
          out_proj(h, heads, t, sharded, o, Wo, Y + (sq * seq + p) * h);
        }
        free(o);
      }
      free(K);
      free(V);
      free(Q);
    }
    return 0;
  }
  for (int64_t rr = 0; rr < n; ++rr) {
    const int64_t r = rows[rr], sq = r / seq, pos = r % seq;
    double* K = (double*)malloc(sizeof(double) * (size_t)((pos + 1) * hd_all));
    double* V = (double*)malloc(sizeof(double) * (size_t)((pos + 1) * hd_all));
    double* Q = (double*)malloc(sizeof(double) * (size_t)((pos + 1) * hd_all));
#pragma omp parallel
    {
      double* x = (double*)malloc(sizeof(double) * (size_t)h);
#pragma omp for schedule(static)
      for (int64_t p = 0; p <= pos; ++p) {
        for (int64_t k = 0; k < h; ++k) x[k] = bf(X[(sq * seq + p) * h + k]);
        qkv_row(h, heads, t, x, Wqkv, Q + p * hd_all, K + p * hd_all, V + p * hd_all);
      }
      free(x);
    }
    double* o = (double*)malloc(sizeof(double) * (size_t)(hd_all + pos + 1));
    attend(heads, d, pos, Q + pos * hd_all, K, V, o, o + hd_all);
    out_proj(h, heads, t, sharded, o, Wo, Y + rr * h);
    free(o);
    free(K);
    free(V);
    free(Q);
  }
  return 0;
}

/* ---- the transformer block ----------------------------------------------------------------- */

static void layernorm_d(int64_t h, double eps, const double* z, double* out) {
  double mean = 0.0;
  for (int64_t k = 0; k < h; ++k) mean += z[k];
  mean /= (double)h;
  double var = 0.0;
  for (int64_t k = 0; k < h; ++k) var += (z[k] - mean) * (z[k] - mean);
  var /= (double)h;
  const double inv = 1.0 / sqrt(var + eps);
  for (int64_t k = 0; k < h; ++k) out[k] = (z[k] - mean) * inv;
}

/* MLP of one row (first linear, activation, second linear; the MLP oracle's layouts). */
static void mlp_row(int64_t h, int64_t F, int t, int act, const double* x, const uint16_t* A, const uint16_t* B,
                    double* y, double* H) {
  const int gated = (act == 3 || act == 4);
  const int64_t Fi = F / t;
  for (int64_t f = 0; f < F; ++f) {
    const int64_t i = f / Fi, j = f % Fi;
    if (gated) {
      const double g = dot_w(h, x, A + (i * 2 * Fi + j) * h);
      const double u = dot_w(h, x, A + (i * 2 * Fi + Fi + j) * h);
      H[f] = oracle_glu(act, g, u);
    } else {
      H[f] = oracle_act(act, dot_w(h, x, A + f * h));
    }
  }
  for (int64_t c = 0; c < h; ++c) {
    double s = 0.0;
    for (int64_t f = 0; f < F; ++f) s += H[f] * bf(B[(f / Fi) * h * Fi + c * Fi + (f % Fi)]);
    y[c] = s;
  }
}

int oracle_block_fwd_bf16(int L, int64_t M, int64_t h, int64_t F, int heads, int64_t seq, int t, int act,
                          double eps, const uint16_t* Z0, const uint16_t* Wqkv, const uint16_t* Wo,
                          const uint16_t* A, const uint16_t* B, const int64_t* seqs, int64_t n_seqs, int64_t upto,
                          double* Zout) {
  if (L < 0 || !attn_shape_ok(M, h, heads, seq, t) || F <= 0 || F % t != 0 || act < 0 || act > 4) return -1;
  if (upto < 0 || upto > seq) return -1;
  const int gated = (act == 3 || act == 4);
  const int64_t d = h / heads, hd_all = heads * d;
  const int64_t qkv_layer = 3 * hd_all * h, o_layer = h * hd_all;
  const int64_t a_layer = (gated ? 2 * F : F) * h, b_layer = h * F;
  const int64_t nseq = M / seq, n = seqs ? n_seqs : nseq;
  for (int64_t ss = 0; ss < n; ++ss)
    if (seqs && (seqs[ss] < 0 || seqs[ss] >= nseq)) return -2;
  double* Z = (double*)malloc(sizeof(double) * (size_t)(upto * h));
  double* Q = (double*)malloc(sizeof(double) * (size_t)(upto * hd_all));
  double* K = (double*)malloc(sizeof(double) * (size_t)(upto * hd_all));
  double* V = (double*)malloc(sizeof(double) * (size_t)(upto * hd_all));
  for (int64_t ss = 0; ss < n; ++ss) {
    const int64_t sq = seqs ? seqs[ss] : ss;
    for (int64_t p = 0; p < upto; ++p)
      for (int64_t k = 0; k < h; ++k) Z[p * h + k] = bf(Z0[(sq * seq + p) * h + k]);
    for (int l = 0; l < L; ++l) {
      const uint16_t* Wqkv_l = Wqkv + l * qkv_layer;
      const uint16_t* Wo_l = Wo + l * o_layer;
      /* attention sublayer: Z += Attn(LN(Z)) */
#pragma omp parallel
      {
        double* ln = (double*)malloc(sizeof(double) * (size_t)h);
#pragma omp for schedule(static)
        for (int64_t p = 0; p < upto; ++p) {
          layernorm_d(h, eps, Z + p * h, ln);
          qkv_row(h, heads, t, ln, Wqkv_l, Q + p * hd_all, K + p * hd_all, V + p * hd_all);
        }
        free(ln);
      }
#pragma omp parallel
      {
        double* o = (double*)malloc(sizeof(double) * (size_t)(hd_all + upto + h));
        double* w = o + hd_all;
        double* y = w + upto;
#pragma omp for schedule(dynamic, 1)
        for (int64_t p = 0; p < upto; ++p) {
          attend(heads, d, p, Q + p * hd_all, K, V, o, w);
          out_proj(h, heads, t, 0, o, Wo_l, y);
          /* rows are updated after every row's keys and values were formed from the old Z */
          for (int64_t k = 0; k < h; ++k) Z[p * h + k] += y[k];
        }
        free(o);
      }
      /* MLP sublayer: Z += MLP(LN(Z)) */
#pragma omp parallel
      {
        double* buf = (double*)malloc(sizeof(double) * (size_t)(2 * h + F));
        double* ln = buf;
        double* y = buf + h;
        double* H = buf + 2 * h;
#pragma omp for schedule(static)
        for (int64_t p = 0; p < upto; ++p) {
          layernorm_d(h, eps, Z + p * h, ln);
          mlp_row(h, F, t, act, ln, A + l * a_layer, B + l * b_layer, y, H);
          for (int64_t k = 0; k < h; ++k) Z[p * h + k] += y[k];
        }
        free(buf);
      }
    }
    memcpy(Zout + ss * upto * h, Z, sizeof(double) * (size_t)(upto * h));
  }
  free(Z);
  free(Q);
  free(K);
  free(V);
  return 0;
}
