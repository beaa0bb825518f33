/*
 * oracle.h -- CPU oracle for the chunked tensor-parallel MLP and attention (test infrastructure).
 *
 * This library is test infrastructure.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or constant
 * with the CUDA library; neither includes nor links the other.
 *
 * It computes, in double precision from the exact values of the bf16 inputs, the plain
 * definition of what the method reaches:
 *
 *   Y = sum_{i<t} act(X . A_i^T) . B_i^T              (forward of one MLP)
 *
 * which is the Megatron-style tensor-parallel MLP (first linear column-parallel, second
 * row-parallel; the sum over shards is what the AllReduce delivers).  Sources:
 *
 *   [Domino]  "DeepSpeed-Domino 深度解析：通过通用张量切分与计算通信重叠实现单机与多节点统一的
 *             LLM 张量并行训练" -- section "TP 的数据依赖：通信为何难以隐藏" (a layer is XAB=Y
 *             followed by AllReduce(Y); for the MLP both A and B are linears), section
 *             "Domino 核心设计：三种张量切分策略" (row split of X, column split of B, 2D),
 *             section "实现与优化" (forward: GeMM + GeLU + GeMM, Dropout/Residual/LayerNorm;
 *             backward: each grad matmul is an input-gradient GEMM plus a weight-gradient GEMM).
 *   [Primer]  nxmr.cn article on DP/TP/PP -- section "3.1 TP的切分方式与计算模式": column split
 *             X[A1,A2] = [XA1, XA2]; row split X[A1;A2] = XA1 + XA2 (partial sums to reduce).
 *   [Overlap] "04 · TP/SP 的通信-计算 overlap 与工程优化" -- section "1. 粗粒度：dgrad 通信 ∥
 *             wgrad 计算" (dgrad = grad_output . weight, wgrad = grad_output^T . input,
 *             accumulated into an fp32 main_grad).
 *
 * Storage (row-major, nn.Linear [out, in]):
 *   X  : M x h.   A : t shards; shard i is F_i x h, or for gated activations 2F_i x h
 *        (F_i gate rows, then F_i up rows).   B : t shards; shard i is h x F_i.
 *   F_i = F / t.  The unsharded first weight is the row concatenation of the A shards;
 *   the unsharded second weight is the column concatenation Bfull[c, i*F_i + j] = B_i[c, j].
 *
 * Activations (act):  0 none, 1 relu, 2 gelu (erf form), 3 swiglu (silu(gate) * up),
 *   4 bilinear (gate * up; a gated form whose integer inputs give integer outputs).
 *
 * Every function returns 0 on success and a negative value on invalid sizes.
 * Row and feature selections let callers evaluate samples of large problems; rows are
 * independent in every function, so a sample equals the same rows of the full result.
 */
#ifndef ORACLE_H
#define ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Forward.  rows[n_rows] selects output rows (NULL: all M rows, n_rows ignored).
 * sharded = 0: Y[r,c] = sum over the unsharded ffn index f of H[r,f] * Bfull[c,f].
 * sharded = 1: each shard's partial P_i = H_i . B_i^T is formed and Y = ((P_0+P_1)+...)+P_{t-1}.
 * Y: n_rows x h doubles.  H_out (nullable): n_rows x F doubles, the activation output. */
int oracle_mlp_fwd_bf16(int64_t M, int64_t h, int64_t F, int t, int act,
                        const uint16_t* X, const uint16_t* A, const uint16_t* B,
                        const int64_t* rows, int64_t n_rows, int sharded,
                        double* Y, double* H_out);
int oracle_mlp_fwd_f64(int64_t M, int64_t h, int64_t F, int t, int act,
                       const double* X, const double* A, const double* B,
                       const int64_t* rows, int64_t n_rows, int sharded,
                       double* Y, double* H_out);

/* Backward of one MLP for output gradient gY (M x h).
 * dX (nullable): n_rows x h, gradient w.r.t. X at the selected rows.
 * feats[n_feats] selects unsharded ffn indices f (NULL: all F).
 * dA (nullable): n_feats x R x h, R = 2 for gated (gate row then up row of feature f), else 1.
 * dB (nullable): n_feats x h, dB[ff][c] = dL/dBfull[c, f].
 * The weight gradients sum over all M rows. */
int oracle_mlp_bwd_bf16(int64_t M, int64_t h, int64_t F, int t, int act,
                        const uint16_t* X, const uint16_t* A, const uint16_t* B, const uint16_t* gY,
                        const int64_t* rows, int64_t n_rows, double* dX,
                        const int64_t* feats, int64_t n_feats, double* dA, double* dB);
int oracle_mlp_bwd_f64(int64_t M, int64_t h, int64_t F, int t, int act,
                       const double* X, const double* A, const double* B, const double* gY,
                       const int64_t* rows, int64_t n_rows, double* dX,
                       const int64_t* feats, int64_t n_feats, double* dA, double* dB);

/* LayerNorm without affine parameters: (z - mean) / sqrt(var + eps), biased variance. */
int oracle_layernorm_bf16(int64_t M, int64_t h, double eps, const uint16_t* Z,
                          const int64_t* rows, int64_t n_rows, double* out);
int oracle_layernorm_f64(int64_t M, int64_t h, double eps, const double* Z,
                         const int64_t* rows, int64_t n_rows, double* out);

/* Pre-LN residual stack of L layers: Z_{l+1} = Z_l + MLP_l(LN(Z_l)).
 * A: L consecutive layer blocks of the A storage; B likewise.  Zout: n_rows x h. */
int oracle_stack_fwd_bf16(int L, int64_t M, int64_t h, int64_t F, int t, int act, double eps,
                          const uint16_t* Z0, const uint16_t* A, const uint16_t* B,
                          const int64_t* rows, int64_t n_rows, double* Zout);

/* Backward of the pre-LN residual stack for the gradient gZL of Z_L: gZ0 (n_rows x h) is the
 * gradient w.r.t. the stack input at the selected rows.  dA, dB (nullable; then rows must be
 * NULL): the weight gradients of every layer, summed over all M rows, in the A and B storage
 * layouts (L layer blocks each).  Returns -3 if weight gradients are asked for a row subset. */
int oracle_stack_bwd_bf16(int L, int64_t M, int64_t h, int64_t F, int t, int act, double eps,
                          const uint16_t* Z0, const uint16_t* A, const uint16_t* B, const uint16_t* gZL,
                          const int64_t* rows, int64_t n_rows, double* gZ0, double* dA, double* dB);
int oracle_stack_bwd_f64(int L, int64_t M, int64_t h, int64_t F, int t, int act, double eps,
                         const double* Z0, const double* A, const double* B, const double* gZL,
                         const int64_t* rows, int64_t n_rows, double* gZ0, double* dA, double* dB);

/* Attention sublayer (oracle_attn.c): causal multi-head self-attention within sequences of `seq`
 * tokens (M % seq == 0, token r at position r % seq), heads split over t shards, then the output
 * projection; Y (n_rows x h) = sum over heads of attention(X) . Wo^T, no residual.  sharded = 1
 * forms each shard's partial and sums them in shard order.  Layouts in oracle_attn.c. */
int oracle_attn_fwd_bf16(int64_t M, int64_t h, int heads, int64_t seq, int t, const uint16_t* X,
                         const uint16_t* Wqkv, const uint16_t* Wo, const int64_t* rows, int64_t n_rows,
                         int sharded, double* Y);

/* Pre-LN transformer block stack (oracle_attn.c), L layers of
 *   Z += Attn(LN(Z));  Z += MLP(LN(Z))
 * evaluated for the sequences seqs[n_seqs] (NULL: all M / seq), positions 0 .. upto-1 of each
 * (causality makes the prefix independent of later positions).  Zout: n_seqs x upto x h.
 * Per-layer weights: Wqkv (3h x h as t shards), Wo (h x h as t shards), A and B as the MLP. */
int oracle_block_fwd_bf16(int L, int64_t M, int64_t h, int64_t F, int heads, int64_t seq, int t, int act,
                          double eps, const uint16_t* Z0, const uint16_t* Wqkv, const uint16_t* Wo,
                          const uint16_t* A, const uint16_t* B, const int64_t* seqs, int64_t n_seqs,
                          int64_t upto, double* Zout);

/* FP8 variant of the MLP forward (oracle_fp8.c): E4M3 operands X8 (M x h), A8, B8 (the MLP
 * layouts) with per-tensor scales sx, sa, sb; H re-quantised to E4M3 with scale sh; Y (n_rows x h)
 * = sh sb (H8 . B8^T) in double.  H8_out (nullable): the n_rows x F codes of H8. */
int oracle_mlp_fwd_fp8(int64_t M, int64_t h, int64_t F, int t, int act, const uint8_t* X8, const uint8_t* A8,
                       const uint8_t* B8, double sx, double sa, double sb, double sh, const int64_t* rows,
                       int64_t n_rows, double* Y, uint8_t* H8_out);
/* E4M3 code <-> value: decode exactly; encode an fp32 value to the nearest, ties to even, saturating
 * at +-448; NaN -> 0x7F. */
double oracle_e4m3_decode(uint8_t code);
uint8_t oracle_e4m3_encode(double x);

/* Elementwise helpers, exposed so tests can pin them against special values. */
double oracle_act(int act, double z);        /* non-gated activations */
double oracle_act_grad(int act, double z);
double oracle_glu(int act, double g, double u);  /* gated activations */
double oracle_glu_dg(int act, double g, double u);
double oracle_glu_du(int act, double g, double u);

int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
