// kernels.h -- host-side interface between the C-ABI layer (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

namespace dm {

// Devices a process may drive; launch facts (shared-memory opt-in, co-resident grid) are cached
// per device ordinal below this bound.
constexpr int kMaxDevices = 64;

// Activation codes (same values as domino_act).
enum : int { ACT_NONE = 0, ACT_RELU = 1, ACT_GELU = 2, ACT_SWIGLU = 3, ACT_BILINEAR = 4 };

// GEMM tile shape: each CTA holds a 128 x 256 fp32 accumulator in TMEM per tile; the K loop
// moves 64 bf16 (128 bytes, one swizzle atom) per pipeline stage.  With kPairMma a CTA pair
// (cluster of 2) computes a 256 x 256 tile with tcgen05.mma.cta_group::2, each CTA staging
// its own 128 rows of A and 128 rows of B.
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr bool kPairMma = true;
constexpr int kTileM = kPairMma ? 2 * kBM : kBM;   // rows of D per tile
constexpr int kBBoxRows = kPairMma ? 128 : 256;     // TMA box height of a K-major B operand

// Epilogues (what happens to the fp32 accumulator tile D).
enum GemmEpi : int {
  EPI_ACT_BF16 = 0,  // out0 = bf16(act(D));  out1 (nullable) = bf16(D)
  EPI_GLU_BF16 = 1,  // D = [gate(128) | up(128)]: out0 = bf16(glu); out1 (nullable): gate at +0, up at +off1
  EPI_F32_STORE = 2, // out0 = D (fp32)
  EPI_F32_ACCUM = 3, // out0 += D (fp32)
  EPI_ACT_BWD = 4,   // in0 = Z: out0 = bf16(D * act'(Z)); out1 = bf16(act(Z))
  EPI_GLU_BWD = 5,   // in0: G at +0, U at +offi: out0: dG at +0, dU at +off0; out1 = bf16(glu(G, U))
  EPI_F32_REDUCE = 6, // batch g = shard, the shards of a tile in order: S = P_0, S += P_g (fp32, held
                      //   on chip); then out1 = bf16(in0 + S) (residual in0 nullable)
  EPI_ACT_F8 = 7,     // FP8 operands: out0 = e4m3(act(alpha D) * out_scale)
  EPI_GLU_F8 = 8,     // FP8 operands, D = [gate | up]: out0 = e4m3(glu(alpha gate, alpha up) * out_scale)
};

// The kernel instantiations the library uses.  A/B operand majorness: K = K-major
// (contiguous along the reduction dim), MN = contiguous along rows/cols of D.
enum GemmVariant : int {
  GV_FWD_ACT = 0,     // first linear, non-gated:     EPI_ACT_BF16,  A K, B K
  GV_FWD_GLU = 1,     // first linear, gated:         EPI_GLU_BF16,  A K, B K (gate/up 4-D map)
  GV_FWD_PARTIAL = 2, // second linear -> partials:   EPI_F32_STORE, A K, B K
  GV_BWD_ACT = 3,     // dH with act backward:        EPI_ACT_BWD,   A K, B MN
  GV_BWD_GLU = 4,     // dH with gated backward:      EPI_GLU_BWD,   A K, B MN
  GV_BWD_PARTIAL = 5, // dX partials:                 EPI_F32_STORE, A K, B MN
  GV_WGRAD = 6,       // weight gradients (+=):       EPI_F32_ACCUM, A MN, B MN
  GV_FWD_REDUCE = 7,  // second linear + shard-sum:   EPI_F32_REDUCE, A K, B K
  GV_BWD_REDUCE = 8,  // dX partials + shard-sum:     EPI_F32_REDUCE, A K, B MN
  // FP8 (E4M3) operands, fp32 accumulation (gemm_fp8.cu); the fp32 epilogues scale D by alpha
  GV_F8_FWD_ACT = 9,      // first linear, non-gated -> E4M3 H:  EPI_ACT_F8
  GV_F8_FWD_GLU = 10,     // first linear, gated -> E4M3 H:      EPI_GLU_F8
  GV_F8_FWD_PARTIAL = 11, // second linear -> fp32 partials:     EPI_F32_STORE
  GV_F8_FWD_REDUCE = 12,  // second linear + shard-sum:          EPI_F32_REDUCE
  GV_COUNT = 13
};

// Per-launch GEMM description.  D[g] (M x N per batch g) = A_op[g] . B_op[g]^T.
// TMA coordinates: K-major operand (k, row + row_off, g * bmul); MN-major (row + row_off, k, g * bmul);
// the gated first-linear B operand uses a 4-D map (k, row, half, g).
struct GemmArgs {
  int32_t batches, m_tiles, n_tiles, k_blocks;
  int32_t M, N;
  int32_t a_row_off, a_bmul;
  int32_t b_row_off, b_bmul;
  int32_t act;
  int32_t err_site;
  int32_t cross_batch;  // tile order: 0 = batch after batch; 1 = the batches side by side along N (below)
  float alpha;      // FP8 variants: scale of the accumulator (product of the operand scales)
  float out_scale;  // EPI_ACT_F8 / EPI_GLU_F8: factor applied before the E4M3 rounding (1 / sh)
  void* out0;
  int64_t ld0, bs0, off0;
  void* out1;
  int64_t ld1, bs1, off1;
  const void* in0;
  int64_t ldi, bsi, offi;
  // fused shard-sum only: scratch for the shard split of the last round of output tiles (partial
  // slots of 256 KiB, then one 32-bit counter per slot), `part_bytes` long (0: no split).  The
  // launcher sets `split` (units sharing each tile of that round, 1 = none) and `flags`.
  void* part;
  int64_t part_bytes;
  uint32_t* flags;
  int32_t split;
};

int gemm_out_tile_n(int variant);  // 128 for GV_FWD_GLU, else 256

// Launch one GEMM; the grid (persistent: one CTA or CTA pair per SM or SM pair) is chosen here.
// Tensor maps of the epilogues that move their data with TMA (box 32 x 32 elements):
//  fp32-partial variants (GV_FWD_PARTIAL, GV_BWD_PARTIAL): m[0] = fp32 output (N, M, batches),
//    128-byte swizzle.
//  activation-backward variants (GV_BWD_ACT, GV_BWD_GLU), all bf16 with 64-byte swizzle and
//    (F_i, M, shards) extents: m[0] saved Z or G (read), m[1] saved U (read, gated),
//    m[2] dZ or dG (written), m[3] dU (written, gated), m[4] recomputed H (written).
//  Other variants ignore the maps.
struct EpiMaps {
  CUtensorMap m[5];
};

cudaError_t launch_gemm_fwd(int variant, const CUtensorMap& ta, const CUtensorMap& tb, const EpiMaps& em,
                            const GemmArgs& args, cudaStream_t st);
cudaError_t launch_gemm_bwd(int variant, const CUtensorMap& ta, const CUtensorMap& tb, const EpiMaps& em,
                            const GemmArgs& args, cudaStream_t st);
// FP8 variants (GV_F8_*); operand maps are uint8 with 128-element (128-byte) K boxes, and
// args.k_blocks counts 128-element K steps.
cudaError_t launch_gemm_fp8(int variant, const CUtensorMap& ta, const CUtensorMap& tb, const EpiMaps& em,
                            const GemmArgs& args, cudaStream_t st);
// Self-test of the bounded-wait failure path (see domino_selftest_wait_timeout).
cudaError_t launch_wait_selftest(uint64_t timeout_ns, int site, cudaStream_t st);
// Reads and clears the device error word of the GEMM kernels in each translation unit.
cudaError_t take_gemm_fwd_error(int* code);
cudaError_t take_gemm_bwd_error(int* code);
cudaError_t take_gemm_fp8_error(int* code);

// Causal multi-head self-attention of one row chunk (attention.cu), head dimension 128.  QKV: the
// fused projection output, per token the t shards' [query heads | key heads | value heads], head
// slot (shard * 3 + which) * nhi + local head; O: per token the heads in global order.  Maps:
// tm_qkv 4-D (128, 3 * heads, seq, sequences), box (64, 1, 128, 1); tm_o 4-D (128, heads, seq,
// sequences), box (64, 1, 32, 1); both bf16 with 128-byte swizzle.
struct AttnArgs {
  int32_t seq;       // tokens per sequence
  int32_t heads;     // heads in total
  int32_t nhi;       // heads per shard
  int32_t n_qblk;    // query blocks of 128 per sequence
  float scale_log2;  // log2(e) / sqrt(head dimension)
  int32_t err_site;
};
// max_ctas: grid cap of the persistent kernel (0 = one CTA per SM).
cudaError_t launch_attention(const CUtensorMap& tm_qkv, const CUtensorMap& tm_o, const AttnArgs& a, int nseq,
                             int max_ctas, cudaStream_t st);
cudaError_t take_attn_error(int* code);

// Shard-sum (AllReduce stand-in) and LayerNorm.
cudaError_t launch_shard_sum(const float* P, int t, int64_t rows, int64_t cols,
                             const uint16_t* res, int64_t ld_res, uint16_t* Y, int64_t ld_y,
                             int grid_cap, cudaStream_t st);
// Same grid as launch_shard_sum, no reduction: copies res into Y when res is given, else does
// nothing (the timing stand-in of domino_debug_skip_reduce).
cudaError_t launch_noreduce(int64_t rows, int64_t cols, const uint16_t* res, int64_t ld_res, uint16_t* Y,
                            int64_t ld_y, int grid_cap, cudaStream_t st);
cudaError_t launch_layernorm(const uint16_t* Z, int64_t rows, int64_t h, float eps, uint16_t* out,
                             float* rstd, cudaStream_t st);
cudaError_t launch_act_eval(int act, const float* a, const float* b, float* out, float* da, float* db, int64_t n,
                            cudaStream_t st);
cudaError_t launch_layernorm_bwd(const uint16_t* gN, const uint16_t* N, const float* rstd, const uint16_t* res,
                                 uint16_t* out, int64_t rows, int64_t h, cudaStream_t st);

// Tensor maps (zero fill out of bounds).  dims[0] is innermost; strides_bytes[i] is the stride of
// dims[i+1].  elem_bytes: 1 = 8-bit codes, 2 = bf16, 4 = fp32.  swizzle_bytes: 128 or 64.
bool tma_encoder_ready(std::string* err);
bool make_map(CUtensorMap* map, int elem_bytes, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides_bytes, const uint32_t* box, std::string* err, int swizzle_bytes = 128);
inline bool make_map_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides_bytes, const uint32_t* box, std::string* err) {
  return make_map(map, 2, base, rank, dims, strides_bytes, box, err);
}

}  // namespace dm
