// api.cu -- the C ABI (include/domino.h): argument validation, workspace layout, TMA maps and
// the chunk scheduler that pipelines the shard-sum of chunk k (reduction stream) against the
// GEMMs of chunk k+1 (compute stream); a call's last chunk, which has no chunk k+1, is reduced
// inside its GEMM.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/domino.h"
#include "kernels.h"

using dm::GemmArgs;

struct TimedLaunch {
  int kind;
  cudaEvent_t a, b;
};

struct domino_handle_s {
  int device = 0;
  int num_sms = 0;
  cudaStream_t s_comp = nullptr;  // GEMMs, LayerNorm
  cudaStream_t s_red = nullptr;   // shard-sums (the AllReduce stand-in)
  cudaEvent_t ev_fork = nullptr, ev_join_c = nullptr, ev_join_r = nullptr;
  cudaEvent_t ev_part[2] = {nullptr, nullptr};  // partial slot s written (compute -> reduce)
  cudaEvent_t ev_red[2] = {nullptr, nullptr};   // partial slot s consumed (reduce -> compute)
  std::vector<cudaEvent_t> ev_row;              // row chunk j of the previous layer reduced
  bool timing = false;
  std::vector<TimedLaunch> timed;
  std::vector<cudaEvent_t> timing_pool;
  int64_t launches = 0;
  int64_t fail_countdown = 0;  // > 0: the launch attempt that brings it to 0 fails (test hook)
  bool skip_reduce = false;    // timing hook: shard-sums replaced by a kernel that does no reduction
};

namespace {

thread_local std::string t_last_error;

domino_status fail(domino_status s, const std::string& msg) {
  t_last_error = msg;
  return s;
}

domino_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DOMINO_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define DM_CUDA(call, what)                     \
  do {                                          \
    const cudaError_t e_ = (call);              \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

constexpr size_t kAlign = 1024;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
// NVTX ranges (header-only NVTX v3: no cost unless a profiler is attached) around every entry
// point, row chunk and kernel enqueue, so a timeline shows the schedule.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

struct NvtxChunk {
  explicit NvtxChunk(int pc) {
    char b[32];
    std::snprintf(b, sizeof b, "row chunk %d", pc);
    nvtxRangePushA(b);
  }
  ~NvtxChunk() { nvtxRangePop(); }
  NvtxChunk(const NvtxChunk&) = delete;
  NvtxChunk& operator=(const NvtxChunk&) = delete;
};

const char* kernel_kind_name(int kind) {
  static const char* const names[DOMINO_K_COUNT] = {"gemm_fwd1", "gemm_fwd2", "shard_sum", "layernorm",
                                                     "gemm_dgrad_h", "gemm_wgrad_b", "gemm_dgrad_x", "gemm_wgrad_a",
                                                     "layernorm_bwd", "gemm_qkv", "attention", "gemm_oproj"};
  return (kind >= 0 && kind < DOMINO_K_COUNT) ? names[kind] : "kernel";
}

bool gated(int act) { return act == DOMINO_ACT_SWIGLU || act == DOMINO_ACT_BILINEAR; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// CTA pairs a GB300 keeps resident for the GEMMs (152 SMs); the workspace is sized for it, and the
// launcher skips the fused shard split on a device whose count needs more (a host-only size query
// cannot ask the device).
constexpr int kGb300Pairs = 76;

// Scratch of the fused shard-sum's shard split (the launcher in gemm.cuh) for an m x n output of t
// shards on `units` CTA pairs: a partial slot of 256 x 256 fp32 per shard of each tile of a last
// round of at most half as many tiles as units (or of every tile when there are fewer tiles than
// units), then a 32-bit counter per slot; 0 when no round is split.
size_t fused_split_bytes(int64_t m, int64_t n, int t, int units) {
  const int64_t tiles = cdiv(m, dm::kTileM) * cdiv(n, dm::kBN);
  if (tiles == 0 || t < 2) return 0;
  const int64_t u = tiles < units ? std::min<int64_t>(tiles * t, units) : units;
  const int64_t rest = tiles % u;
  if (rest == 0 || u / rest < 2) return 0;
  return size_t(rest * t) * (size_t(dm::kTileM) * dm::kBN * 4 + 4);
}

struct Plan {
  int64_t M, h, F, Fi, m, n, a_rows, Ri;
  int t, p, q, act, sched, layers, nslots;
  int heads = 0, seq = 0;  // attention passes
  int reduce_ctas = 0;     // shard-sum grid cap, 0 = default
  int attn_ctas = 0;       // attention grid cap, 0 = one CTA per SM
  float eps;
  bool gated;
  // workspace offsets
  size_t off_h = 0, off_ln = 0, off_dz = 0, off_hb = 0, off_gn = 0, off_part = 0, part_slot = 0, total = 0;
  size_t off_qkv = 0, off_o = 0;  // attention: fused projection output (m x 3h), attention output (m x h)
  // layer-stack save buffer (training forward -> backward): per layer the LayerNorm output N
  // (M x h bf16), the first-linear output (M x a_rows bf16) and 1/sqrt(var + eps) (M fp32)
  size_t save_n = 0, save_act = 0, save_rstd = 0, save_layer = 0;
};

domino_status make_plan_impl(const domino_cfg* c, int pass, Plan* P) {
  if (!c) return fail(DOMINO_ERR_INVALID_ARG, "cfg is NULL");
  if (c->flags != 0) return fail(DOMINO_ERR_INVALID_ARG, "cfg->flags must be 0");
  if (c->reduce_ctas < 0) return fail(DOMINO_ERR_INVALID_ARG, "cfg->reduce_ctas must be >= 0");
  if (c->attn_ctas < 0) return fail(DOMINO_ERR_INVALID_ARG, "cfg->attn_ctas must be >= 0");
  if (c->M < 0 || c->h <= 0 || (pass != DOMINO_PASS_ATTN && c->ffn <= 0) || c->t < 1 || c->p < 1 || c->q < 1)
    return fail(DOMINO_ERR_INVALID_ARG, "need M >= 0, h > 0, ffn > 0, t >= 1, p >= 1, q >= 1");
  if (c->act < DOMINO_ACT_NONE || c->act > DOMINO_ACT_BILINEAR)
    return fail(DOMINO_ERR_INVALID_ARG, "unknown activation");
  if (c->sched < DOMINO_SCHED_SERIAL || c->sched > DOMINO_SCHED_FUSED)
    return fail(DOMINO_ERR_INVALID_ARG, "unknown schedule");
  if (c->M % c->p != 0) return fail(DOMINO_ERR_INVALID_ARG, "M must be divisible by p");
  if (c->h % c->q != 0) return fail(DOMINO_ERR_INVALID_ARG, "h must be divisible by q");
  const bool attn = pass == DOMINO_PASS_ATTN || pass == DOMINO_PASS_BLOCK;
  const bool mlp = pass != DOMINO_PASS_ATTN;
  if (mlp && c->ffn % c->t != 0) return fail(DOMINO_ERR_INVALID_ARG, "ffn must be divisible by t");
  const int64_t Fi = mlp ? c->ffn / c->t : 8;
  if (c->h % 8 != 0 || Fi % 8 != 0 || (c->h / c->q) % 8 != 0)
    return fail(DOMINO_ERR_ALIGNMENT, "h, ffn/t and h/q must be multiples of 8 (16-byte rows)");
  if (pass == DOMINO_PASS_FWD_FP8 && (c->h % 16 != 0 || Fi % 16 != 0))
    return fail(DOMINO_ERR_ALIGNMENT, "FP8: h and ffn/t must be multiples of 16 (16-byte rows)");
  if (attn) {
    if (c->heads < 1 || c->seq < 1) return fail(DOMINO_ERR_INVALID_ARG, "attention needs heads >= 1 and seq >= 1");
    if (c->h % c->heads != 0 || c->heads % c->t != 0)
      return fail(DOMINO_ERR_INVALID_ARG, "need h % heads == 0 and heads % t == 0");
    if (c->h / c->heads != 128) return fail(DOMINO_ERR_UNSUPPORTED, "head dimension h / heads must be 128");
    if ((c->M / c->p) % c->seq != 0)
      return fail(DOMINO_ERR_INVALID_ARG, "row chunks must hold whole sequences: M % (p * seq) == 0");
    // work units of one attention launch (pairs of query-block pairs x heads x sequences) must
    // fit a 32-bit index
    const int64_t n_qblk = cdiv(c->seq, 128), units = ((n_qblk + 1) / 2 + 1) / 2 * c->heads * ((c->M / c->p) / c->seq);
    if (units > (int64_t(1) << 31) - 1)
      return fail(DOMINO_ERR_UNSUPPORTED, "more attention work per row chunk than one launch covers");
  }
  if (c->M > (int64_t(1) << 31) - 1 || c->h > (int64_t(1) << 20) || c->ffn > (int64_t(1) << 24))
    return fail(DOMINO_ERR_UNSUPPORTED, "size beyond the supported range");
  // one shard-sum launch covers m x n outputs as 16-byte vectors counted in 32 bits (see
  // domino_shard_sum)
  if ((c->M / c->p) * ((c->h / c->q) / 8) >= (int64_t(1) << 31))
    return fail(DOMINO_ERR_UNSUPPORTED, "row chunk x column chunk too large for one reduction launch");
  if (pass == DOMINO_PASS_STACK || pass == DOMINO_PASS_STACK_BWD) {
    if (c->layers < 1) return fail(DOMINO_ERR_INVALID_ARG, "layers must be >= 1");
    if (!(c->ln_eps > 0.0f)) return fail(DOMINO_ERR_INVALID_ARG, "ln_eps must be > 0");
  }
  if (pass < DOMINO_PASS_FWD || pass > DOMINO_PASS_FWD_FP8) return fail(DOMINO_ERR_INVALID_ARG, "bad pass");
  if (pass == DOMINO_PASS_BLOCK) {
    if (c->layers < 1) return fail(DOMINO_ERR_INVALID_ARG, "layers must be >= 1");
    if (!(c->ln_eps > 0.0f)) return fail(DOMINO_ERR_INVALID_ARG, "ln_eps must be > 0");
  }
  Plan& p = *P;
  p.M = c->M; p.h = c->h; p.F = c->ffn; p.Fi = Fi; p.t = c->t; p.p = c->p; p.q = c->q;
  p.act = c->act; p.sched = c->sched; p.layers = c->layers; p.eps = c->ln_eps;
  p.reduce_ctas = c->reduce_ctas;
  p.attn_ctas = c->attn_ctas;
  if (attn) {
    p.heads = c->heads;
    p.seq = c->seq;
  }
  p.gated = gated(c->act);
  p.m = c->M / c->p;
  p.n = c->h / c->q;
  p.a_rows = p.gated ? 2 * p.F : p.F;
  p.Ri = p.gated ? 2 * Fi : Fi;
  p.nslots = (p.p * p.q >= 2) ? 2 : 1;
  p.save_n = 0;
  p.save_act = align_up(size_t(p.M) * p.h * 2);
  p.save_rstd = p.save_act + align_up(size_t(p.M) * p.a_rows * 2);
  p.save_layer = p.save_rstd + align_up(size_t(p.M) * 4);
  size_t off = 0;
  if (p.M == 0) {
    p.total = 0;
    return DOMINO_OK;
  }
  if (attn) {
    p.off_qkv = off;
    off = align_up(off + size_t(p.m) * 3 * p.h * 2);
    p.off_o = off;
    off = align_up(off + size_t(p.m) * p.h * 2);
    if (pass == DOMINO_PASS_BLOCK) {
      p.off_ln = off;
      off = align_up(off + size_t(p.m) * p.h * 2);
      p.off_h = off;
      off = align_up(off + size_t(p.m) * p.F * 2);
    }
  } else if (pass == DOMINO_PASS_FWD_FP8) {
    p.off_h = off;  // E4M3 first-linear output of one row chunk
    off = align_up(off + size_t(p.m) * p.F);
  } else if (pass == DOMINO_PASS_FWD || pass == DOMINO_PASS_STACK) {
    p.off_h = off;
    off = align_up(off + size_t(p.m) * p.F * 2);
    if (pass == DOMINO_PASS_STACK) {
      p.off_ln = off;
      off = align_up(off + size_t(p.m) * p.h * 2);
    }
  } else {
    p.off_dz = off;
    off = align_up(off + size_t(p.m) * p.a_rows * 2);
    p.off_hb = off;
    off = align_up(off + size_t(p.m) * p.F * 2);
    if (pass == DOMINO_PASS_STACK_BWD) {
      p.off_gn = off;  // gradient at the LayerNorm output, all rows
      off = align_up(off + size_t(p.M) * p.h * 2);
    }
  }
  // partial slots of t x m x n fp32; the fused schedule keeps its sums on chip and needs only the
  // scratch of the shard split of its last round of tiles (fused_split_bytes)
  if (p.sched == DOMINO_SCHED_FUSED) {
    p.nslots = 1;
    p.part_slot = align_up(fused_split_bytes(p.m, p.n, p.t, kGb300Pairs));
  } else {
    p.part_slot = align_up(size_t(p.t) * p.m * p.n * 4);
  }
  p.off_part = off;
  off += p.part_slot * p.nslots;
  p.total = off;
  return DOMINO_OK;
}

// With DOMINO_LOG=1 in the environment every validated plan is printed to stderr: the pass, the
// problem and chunk sizes, the schedule and the workspace layout.
void log_plan(const Plan& P, int pass) {
  const char* v = std::getenv("DOMINO_LOG");
  if (!v || std::strcmp(v, "1") != 0) return;
  static const char* const passes[] = {"fwd", "bwd", "stack", "stack_bwd", "attn", "block", "fwd_fp8"};
  static const char* const scheds[] = {"serial", "intra", "inter", "fused"};
  std::fprintf(stderr,
               "domino plan: pass=%s M=%lld h=%lld ffn=%lld t=%d p=%d q=%d (chunk %lld x %lld) act=%d sched=%s "
               "layers=%d heads=%d seq=%d partial slots=%d x %zu B workspace=%zu B [h@%zu ln@%zu dz@%zu hb@%zu "
               "gn@%zu qkv@%zu o@%zu partials@%zu]\n",
               passes[pass], static_cast<long long>(P.M), static_cast<long long>(P.h), static_cast<long long>(P.F),
               P.t, P.p, P.q, static_cast<long long>(P.m), static_cast<long long>(P.n), P.act, scheds[P.sched],
               P.layers, P.heads, P.seq, P.nslots, P.part_slot, P.total, P.off_h, P.off_ln, P.off_dz, P.off_hb,
               P.off_gn, P.off_qkv, P.off_o, P.off_part);
}

domino_status make_plan(const domino_cfg* c, int pass, Plan* P) {
  const domino_status st = make_plan_impl(c, pass, P);
  if (st == DOMINO_OK) log_plan(*P, pass);
  return st;
}

domino_status check_ws(const Plan& P, void* ws, size_t bytes) {
  if (P.total == 0) return DOMINO_OK;
  if (!ws) return fail(DOMINO_ERR_WORKSPACE, "workspace is NULL");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(DOMINO_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (bytes < P.total)
    return fail(DOMINO_ERR_WORKSPACE, "workspace too small: need " + std::to_string(P.total) + " bytes");
  return DOMINO_OK;
}

domino_status check_ptr(const void* p, const char* name, bool nullable = false) {
  if (!p) {
    if (nullable) return DOMINO_OK;
    return fail(DOMINO_ERR_INVALID_ARG, std::string(name) + " is NULL");
  }
  if (!aligned16(p)) return fail(DOMINO_ERR_ALIGNMENT, std::string(name) + " is not 16-byte aligned");
  return DOMINO_OK;
}

#define DM_TRY(expr)                   \
  do {                                 \
    const domino_status s_ = (expr);   \
    if (s_ != DOMINO_OK) return s_;    \
  } while (0)

// ---- tensor maps --------------------------------------------------------------------------

// 3-D bf16 map: (inner, rows, batch); row stride and batch stride in elements.
domino_status map3(CUtensorMap* m, const void* base, int64_t inner, int64_t rows, int64_t batch,
                   int64_t row_stride, int64_t batch_stride, uint32_t box_inner, uint32_t box_rows) {
  const uint64_t dims[3] = {uint64_t(inner), uint64_t(rows), uint64_t(batch)};
  const uint64_t strides[2] = {uint64_t(row_stride) * 2,
                               uint64_t(batch > 1 ? batch_stride : row_stride * rows) * 2};
  const uint32_t box[3] = {box_inner, box_rows, 1};
  std::string err;
  if (!dm::make_map_bf16(m, base, 3, dims, strides, box, &err)) return fail(DOMINO_ERR_CUDA, err);
  return DOMINO_OK;
}

// K-major operand: box 64 (K) x rows;  MN-major operand: box 64 (M/N) x 64 (K).
domino_status map_k(CUtensorMap* m, const void* base, int64_t K, int64_t rows, int64_t batch,
                    int64_t row_stride, int64_t batch_stride, uint32_t box_rows) {
  return map3(m, base, K, rows, batch, row_stride, batch_stride, 64, box_rows);
}
domino_status map_mn(CUtensorMap* m, const void* base, int64_t MN, int64_t K, int64_t batch,
                     int64_t k_stride, int64_t batch_stride) {
  return map3(m, base, MN, K, batch, k_stride, batch_stride, 64, 64);
}

// bf16 (cols, rows, batch) map with a 32 x 32 box and 64-byte swizzle, for the activation-backward
// epilogue's TMA loads and stores; row and batch strides in elements.
domino_status map_epi_bf16(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t batch,
                           int64_t row_stride, int64_t batch_stride) {
  const uint64_t dims[3] = {uint64_t(cols), uint64_t(rows), uint64_t(batch)};
  const uint64_t strides[2] = {uint64_t(row_stride) * 2, uint64_t(batch > 1 ? batch_stride : row_stride * rows) * 2};
  const uint32_t box[3] = {32, 32, 1};
  std::string err;
  if (!dm::make_map(m, 2, base, 3, dims, strides, box, &err, 64)) return fail(DOMINO_ERR_CUDA, err);
  return DOMINO_OK;
}

// 8-bit (E4M3) K-major operand: (K, rows, batch) with a 128-element (128-byte) K box.
domino_status map_k8(CUtensorMap* m, const void* base, int64_t K, int64_t rows, int64_t batch, int64_t row_stride,
                     int64_t batch_stride, uint32_t box_rows) {
  const uint64_t dims[3] = {uint64_t(K), uint64_t(rows), uint64_t(batch)};
  const uint64_t strides[2] = {uint64_t(row_stride), uint64_t(batch > 1 ? batch_stride : row_stride * rows)};
  const uint32_t box[3] = {128, box_rows, 1};
  std::string err;
  if (!dm::make_map(m, 1, base, 3, dims, strides, box, &err)) return fail(DOMINO_ERR_CUDA, err);
  return DOMINO_OK;
}

// fp32 output map of a partial slot: t contiguous rows x cols blocks, TMA-store box 32 x 32.
domino_status map_f32_out(CUtensorMap* m, const float* base, int64_t cols, int64_t rows, int64_t batch) {
  const uint64_t dims[3] = {uint64_t(cols), uint64_t(rows), uint64_t(batch)};
  const uint64_t strides[2] = {uint64_t(cols) * 4, uint64_t(cols * rows) * 4};
  const uint32_t box[3] = {32, 32, 1};
  std::string err;
  if (!dm::make_map(m, 4, base, 3, dims, strides, box, &err)) return fail(DOMINO_ERR_CUDA, err);
  return DOMINO_OK;
}

// ---- launches -----------------------------------------------------------------------------

cudaEvent_t timing_event(domino_handle H) {
  if (!H->timing_pool.empty()) {
    cudaEvent_t e = H->timing_pool.back();
    H->timing_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

template <class Fn>
domino_status launch(domino_handle H, int kind, cudaStream_t st, const char* what, Fn&& fn) {
  if (H->fail_countdown > 0 && --H->fail_countdown == 0)
    return fail(DOMINO_ERR_CUDA, std::string(what) + ": injected launch failure");
  cudaEvent_t a = nullptr, b = nullptr;
  if (H->timing) {
    a = timing_event(H);
    b = timing_event(H);
    DM_CUDA(cudaEventRecord(a, st), "cudaEventRecord");
  }
  cudaError_t e;
  {
    NvtxRange r(kernel_kind_name(kind));
    e = fn();
  }
  if (e != cudaSuccess) return cuda_fail(e, what);
  H->launches++;
  if (H->timing) {
    DM_CUDA(cudaEventRecord(b, st), "cudaEventRecord");
    H->timed.push_back({kind, a, b});
  }
  return DOMINO_OK;
}

GemmArgs gemm_args(int variant, int batches, int64_t M, int64_t N, int64_t K, int site) {
  GemmArgs a;
  std::memset(&a, 0, sizeof a);
  a.batches = batches;
  a.M = int32_t(M);
  a.N = int32_t(N);
  a.m_tiles = int32_t(cdiv(M, dm::kTileM));
  a.n_tiles = int32_t(cdiv(N, dm::gemm_out_tile_n(variant)));
  a.k_blocks = int32_t(cdiv(K, dm::kBK));
  a.err_site = site << 4;
  a.alpha = 1.0f;
  a.out_scale = 1.0f;
  if (variant >= dm::GV_F8_FWD_ACT) a.k_blocks = int32_t(cdiv(K, 128));  // 128 E4M3 codes per K step
  return a;
}

// `em`: the epilogue's tensor maps (fp32-partial and activation variants); others ignore it.
domino_status run_gemm(domino_handle H, int kind, int variant, const CUtensorMap& ta,
                       const CUtensorMap& tb, const GemmArgs& a, cudaStream_t st,
                       const dm::EpiMaps* em = nullptr) {
  const int64_t tiles = int64_t(a.batches) * a.m_tiles * a.n_tiles;
  if (tiles == 0) return DOMINO_OK;
  const bool needs = variant != dm::GV_WGRAD && variant != dm::GV_F8_FWD_ACT && variant != dm::GV_F8_FWD_GLU &&
                     variant != dm::GV_FWD_REDUCE && variant != dm::GV_BWD_REDUCE && variant != dm::GV_F8_FWD_REDUCE;
  if (needs && em == nullptr) return fail(DOMINO_ERR_INVALID_ARG, "internal: GEMM epilogue without its maps");
  static const dm::EpiMaps kNone = {};
  const dm::EpiMaps& e = em ? *em : kNone;
  const bool fwd_tu = variant <= dm::GV_FWD_PARTIAL || variant == dm::GV_FWD_REDUCE;
  const bool fp8_tu = variant >= dm::GV_F8_FWD_ACT;
  return launch(H, kind, st, "GEMM launch", [&] {
    return fp8_tu   ? dm::launch_gemm_fp8(variant, ta, tb, e, a, st)
           : fwd_tu ? dm::launch_gemm_fwd(variant, ta, tb, e, a, st)
                    : dm::launch_gemm_bwd(variant, ta, tb, e, a, st);
  });
}

// The fused second linear (or input-gradient GEMM) + shard-sum of one column chunk, the sums held
// on chip: `res` (nullable) and `Y` are row-major with leading dimension ld; `scratch` (nullable,
// `scratch_bytes` long) takes the partials of a split last round of tiles (fused_split_bytes).
domino_status run_fused_reduce(domino_handle H, int kind, int variant, const CUtensorMap& ta, const CUtensorMap& tb,
                               GemmArgs a, const uint16_t* res, uint16_t* Y, int64_t ld, void* scratch,
                               size_t scratch_bytes, cudaStream_t st) {
  a.part = scratch;
  a.part_bytes = int64_t(scratch_bytes);
  a.out1 = Y;
  a.ld1 = ld;
  a.in0 = res;
  a.ldi = ld;
  return run_gemm(H, kind, variant, ta, tb, a, st, nullptr);
}

domino_status run_shard_sum(domino_handle H, const float* P, int t, int64_t rows, int64_t cols,
                            const uint16_t* res, int64_t ld_res, uint16_t* Y, int64_t ld_y,
                            int reduce_ctas, cudaStream_t st) {
  const int cap = reduce_ctas > 0 ? reduce_ctas : H->num_sms * 4;
  if (H->skip_reduce)
    return launch(H, DOMINO_K_SHARD_SUM, st, "no-reduce launch",
                  [&] { return dm::launch_noreduce(rows, cols, res, ld_res, Y, ld_y, cap, st); });
  return launch(H, DOMINO_K_SHARD_SUM, st, "shard-sum launch",
                [&] { return dm::launch_shard_sum(P, t, rows, cols, res, ld_res, Y, ld_y, cap, st); });
}

// ---- scheduling helpers ---------------------------------------------------------------------

struct Streams {
  cudaStream_t comp, red;
  bool overlap;
};

domino_status fork(domino_handle H, const Plan& P, cudaStream_t caller, Streams* S) {
  if (H->skip_reduce && P.sched == DOMINO_SCHED_FUSED)
    return fail(DOMINO_ERR_UNSUPPORTED, "domino_debug_skip_reduce applies to the stream schedules, not FUSED");
  // the fused schedule overlaps inside its kernels and runs on the caller's stream
  S->overlap = P.sched != DOMINO_SCHED_SERIAL && P.sched != DOMINO_SCHED_FUSED;
  if (!S->overlap) {
    S->comp = S->red = caller;
    return DOMINO_OK;
  }
  S->comp = H->s_comp;
  S->red = H->s_red;
  DM_CUDA(cudaEventRecord(H->ev_fork, caller), "cudaEventRecord(fork)");
  DM_CUDA(cudaStreamWaitEvent(S->comp, H->ev_fork, 0), "cudaStreamWaitEvent");
  DM_CUDA(cudaStreamWaitEvent(S->red, H->ev_fork, 0), "cudaStreamWaitEvent");
  return DOMINO_OK;
}

domino_status join(domino_handle H, const Streams& S, cudaStream_t caller) {
  if (!S.overlap) return DOMINO_OK;
  DM_CUDA(cudaEventRecord(H->ev_join_c, S.comp), "cudaEventRecord(join)");
  DM_CUDA(cudaEventRecord(H->ev_join_r, S.red), "cudaEventRecord(join)");
  DM_CUDA(cudaStreamWaitEvent(caller, H->ev_join_c, 0), "cudaStreamWaitEvent");
  DM_CUDA(cudaStreamWaitEvent(caller, H->ev_join_r, 0), "cudaStreamWaitEvent");
  return DOMINO_OK;
}

// Joins the internal streams back into the caller's stream whatever the outcome of the schedule,
// so a failed call leaves no dangling work ordering behind; the first error wins.
domino_status finish(domino_handle H, const Streams& S, cudaStream_t caller, domino_status st) {
  if (st == DOMINO_OK) return join(H, S, caller);
  const std::string msg = t_last_error;
  join(H, S, caller);
  t_last_error = msg;
  return st;
}

// Chunk k writes partial slot k % nslots on the compute stream and is reduced on the reduction
// stream; before chunk k + nslots reuses the slot, the compute stream waits for that reduction.
struct SlotRing {
  int64_t k = 0;
  // set by the caller for the call's last chunk: its last reduction has no later GEMM of the call
  // to overlap, so the overlapped schedules fold it into the GEMM (second_linear)
  bool tail = false;
};

domino_status slot_acquire(domino_handle H, const Plan& P, const Streams& S, SlotRing& R, int* slot) {
  *slot = int(R.k % P.nslots);
  if (S.overlap && R.k >= P.nslots)
    DM_CUDA(cudaStreamWaitEvent(S.comp, H->ev_red[*slot], 0), "cudaStreamWaitEvent(slot)");
  return DOMINO_OK;
}

domino_status slot_handoff(domino_handle H, const Streams& S, int slot) {
  if (!S.overlap) return DOMINO_OK;
  DM_CUDA(cudaEventRecord(H->ev_part[slot], S.comp), "cudaEventRecord(part)");
  DM_CUDA(cudaStreamWaitEvent(S.red, H->ev_part[slot], 0), "cudaStreamWaitEvent(part)");
  return DOMINO_OK;
}

domino_status slot_release(domino_handle H, const Streams& S, SlotRing& R, int slot) {
  R.k++;
  if (!S.overlap) return DOMINO_OK;
  DM_CUDA(cudaEventRecord(H->ev_red[slot], S.red), "cudaEventRecord(red)");
  return DOMINO_OK;
}

domino_status ready(domino_handle H) {
  if (!H) return fail(DOMINO_ERR_INVALID_ARG, "handle is NULL");
  int dev = -1;
  DM_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev != H->device) return fail(DOMINO_ERR_INVALID_ARG, "handle belongs to another device");
  // Bind the device's primary context to the calling thread: a thread that has not used CUDA yet
  // (e.g. an autograd worker) has none current, and the tensor-map encoder is a driver-API call.
  DM_CUDA(cudaSetDevice(dev), "cudaSetDevice");
  return DOMINO_OK;
}

// ---- the row-parallel second linear of a sublayer for one row chunk: per column chunk the t shard
// partials P_i = H_i . B_i^T (reduction length Kc per shard) into a partial slot on the compute
// stream and their shard-sum (+ residual res_c) into Yc on the reduction stream, or both in one
// kernel with the fused schedule and for the last column chunk of a call's last row chunk
// (R.tail).  mapH: (Kc, m, t) view of the chunk's shard inputs; mapB: the shards' weights (Kc, h, t).
domino_status second_linear(domino_handle H, const Plan& P, const Streams& S, SlotRing& R, int kind,
                            const CUtensorMap& mapH, const CUtensorMap& mapB, int64_t Kc, float* parts,
                            const uint16_t* res_c, uint16_t* Yc, int site, bool fp8 = false, float alpha = 1.0f) {
  const int v_reduce = fp8 ? dm::GV_F8_FWD_REDUCE : dm::GV_FWD_REDUCE;
  const int v_partial = fp8 ? dm::GV_F8_FWD_PARTIAL : dm::GV_FWD_PARTIAL;
  // column chunk qc with the shard-sum folded into the GEMM; `scratch`: P.part_slot bytes
  auto fused = [&](int qc, void* scratch) {
    GemmArgs a = gemm_args(v_reduce, P.t, P.m, P.n, Kc, site);
    a.a_bmul = 1;
    a.b_row_off = int32_t(qc * P.n);
    a.b_bmul = 1;
    a.alpha = alpha;
    return run_fused_reduce(H, kind, v_reduce, mapH, mapB, a, res_c ? res_c + qc * P.n : nullptr, Yc + qc * P.n,
                            P.h, scratch, P.part_slot, S.comp);
  };
  for (int qc = 0; qc < P.q; ++qc) {
    if (P.sched == DOMINO_SCHED_FUSED) {
      DM_TRY(fused(qc, parts));
      continue;
    }
    int slot;
    DM_TRY(slot_acquire(H, P, S, R, &slot));
    float* part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(parts) + P.part_slot * slot);
    if (S.overlap && R.tail && qc == P.q - 1 && !H->skip_reduce) {
      // The call's last reduction would run with nothing left to overlap: the fused kernel adds the
      // shard partials tile by tile inside the GEMM instead (same order, same single rounding, so the
      // same bits); the slot's memory takes the partials of a split last round of tiles, and it is
      // handed over so that the reduction stream waits for it and the row events and the join that
      // follow on that stream cover it.
      DM_TRY(fused(qc, part));
      DM_TRY(slot_handoff(H, S, slot));
      DM_TRY(slot_release(H, S, R, slot));
      continue;
    }
    GemmArgs a = gemm_args(v_partial, P.t, P.m, P.n, Kc, site);
    a.alpha = alpha;
    a.a_bmul = 1;
    a.b_row_off = int32_t(qc * P.n);
    a.b_bmul = 1;
    a.out0 = part;
    a.ld0 = P.n;
    a.bs0 = P.m * P.n;
    dm::EpiMaps em = {};
    DM_TRY(map_f32_out(&em.m[0], part, P.n, P.m, P.t));
    DM_TRY(run_gemm(H, kind, v_partial, mapH, mapB, a, S.comp, &em));
    DM_TRY(slot_handoff(H, S, slot));
    DM_TRY(run_shard_sum(H, part, P.t, P.m, P.n, res_c ? res_c + qc * P.n : nullptr, P.h,
                         Yc + qc * P.n, P.h, P.reduce_ctas, S.red));
    DM_TRY(slot_release(H, S, R, slot));
  }
  return DOMINO_OK;
}

// ---- forward of one MLP for row chunk pc: first linear into H, then the q column chunks of the
// second linear (second_linear: partial slots reduced on the reduction stream, or fused).
domino_status mlp_chunk_fwd(domino_handle H, const Plan& P, const Streams& S, SlotRing& R,
                            const uint16_t* Xc, const CUtensorMap& mapA, const CUtensorMap& mapB,
                            uint16_t* Hbuf, float* parts, uint16_t* save_c, const uint16_t* res_c,
                            uint16_t* Yc, int site) {
  CUtensorMap mapX, mapH;
  DM_TRY(map_k(&mapX, Xc, P.h, P.m, 1, P.h, 0, 128));
  // first linear: H = act(X_c A^T); gated: per shard, 128 output columns per tile
  {
    const int variant = P.gated ? dm::GV_FWD_GLU : dm::GV_FWD_ACT;
    GemmArgs a = gemm_args(variant, P.gated ? P.t : 1, P.m, P.gated ? P.Fi : P.F, P.h, site);
    a.act = P.act;
    a.cross_batch = 1;  // the shards share X: walk every shard's N-tiles per group of M-tiles
    a.out0 = Hbuf;
    a.ld0 = P.F;
    a.bs0 = P.gated ? P.Fi : 0;
    a.out1 = save_c;
    a.ld1 = P.a_rows;
    a.bs1 = P.gated ? 2 * P.Fi : 0;
    a.off1 = P.Fi;
    // epilogue maps: H (per shard for the gated form), and the saved Z or G, U
    dm::EpiMaps em = {};
    if (P.gated) {
      DM_TRY(map_epi_bf16(&em.m[0], Hbuf, P.Fi, P.m, P.t, P.F, P.Fi));
      if (save_c) {
        DM_TRY(map_epi_bf16(&em.m[1], save_c, P.Fi, P.m, P.t, P.a_rows, P.Ri));
        DM_TRY(map_epi_bf16(&em.m[2], save_c + P.Fi, P.Fi, P.m, P.t, P.a_rows, P.Ri));
      }
    } else {
      DM_TRY(map_epi_bf16(&em.m[0], Hbuf, P.F, P.m, 1, P.F, 0));
      if (save_c) DM_TRY(map_epi_bf16(&em.m[1], save_c, P.F, P.m, 1, P.F, 0));
    }
    DM_TRY(run_gemm(H, DOMINO_K_GEMM_FWD1, variant, mapX, mapA, a, S.comp, &em));
  }
  DM_TRY(map_k(&mapH, Hbuf, P.Fi, P.m, P.t, P.F, P.Fi, 128));
  return second_linear(H, P, S, R, DOMINO_K_GEMM_FWD2, mapH, mapB, P.Fi, parts, res_c, Yc, site + 1);
}

// ---- FP8 forward of one row chunk: the first linear on E4M3 operands with the activation and the
// E4M3 re-quantisation of H (scale 1 / sh) in its epilogue, then the second linear on E4M3 H and B
// into fp32 partials (scaled by sh sb) and their fp32 shard-sum.
domino_status mlp_chunk_fwd_fp8(domino_handle H, const Plan& P, const Streams& S, SlotRing& R, const uint8_t* X8c,
                                const CUtensorMap& mapA, const CUtensorMap& mapB, uint8_t* H8, float* parts,
                                uint16_t* Yc, const float* sc) {
  CUtensorMap mapX, mapH;
  DM_TRY(map_k8(&mapX, X8c, P.h, P.m, 1, P.h, 0, 128));
  {
    const int variant = P.gated ? dm::GV_F8_FWD_GLU : dm::GV_F8_FWD_ACT;
    GemmArgs a = gemm_args(variant, P.gated ? P.t : 1, P.m, P.gated ? P.Fi : P.F, P.h, 10);
    a.act = P.act;
    a.cross_batch = 1;  // the shards share X8
    a.out0 = H8;
    a.ld0 = P.F;
    a.bs0 = P.gated ? P.Fi : 0;
    a.alpha = sc[0] * sc[1];
    a.out_scale = 1.0f / sc[3];
    DM_TRY(run_gemm(H, DOMINO_K_GEMM_FWD1, variant, mapX, mapA, a, S.comp, nullptr));
  }
  DM_TRY(map_k8(&mapH, H8, P.Fi, P.m, P.t, P.F, P.Fi, 128));
  return second_linear(H, P, S, R, DOMINO_K_GEMM_FWD2, mapH, mapB, P.Fi, parts, nullptr, Yc, 11, true,
                       sc[3] * sc[2]);
}

domino_status weight_maps_fp8(const Plan& P, const uint8_t* A8, const uint8_t* B8, CUtensorMap* mapA,
                              CUtensorMap* mapB) {
  if (P.gated) {
    const uint64_t dims[4] = {uint64_t(P.h), uint64_t(P.Fi), 2, uint64_t(P.t)};
    const uint64_t strides[3] = {uint64_t(P.h), uint64_t(P.Fi * P.h), uint64_t(2 * P.Fi * P.h)};
    const uint32_t box[4] = {128, 128, 1, 1};
    std::string err;
    if (!dm::make_map(mapA, 1, A8, 4, dims, strides, box, &err)) return fail(DOMINO_ERR_CUDA, err);
  } else {
    DM_TRY(map_k8(mapA, A8, P.h, P.F, 1, P.h, 0, dm::kBBoxRows));
  }
  DM_TRY(map_k8(mapB, B8, P.Fi, P.h, P.t, P.Fi, P.h * P.Fi, dm::kBBoxRows));
  return DOMINO_OK;
}

domino_status weight_maps_fwd(const Plan& P, const uint16_t* A, const uint16_t* B, CUtensorMap* mapA,
                              CUtensorMap* mapB) {
  if (P.gated) {
    // A shard i = [gate_i ; up_i], each F_i x h: 4-D view (h, F_i, 2, t)
    const uint64_t dims[4] = {uint64_t(P.h), uint64_t(P.Fi), 2, uint64_t(P.t)};
    const uint64_t strides[3] = {uint64_t(P.h) * 2, uint64_t(P.Fi * P.h) * 2, uint64_t(2 * P.Fi * P.h) * 2};
    const uint32_t box[4] = {64, 128, 1, 1};
    std::string err;
    if (!dm::make_map_bf16(mapA, A, 4, dims, strides, box, &err)) return fail(DOMINO_ERR_CUDA, err);
  } else {
    DM_TRY(map_k(mapA, A, P.h, P.F, 1, P.h, 0, dm::kBBoxRows));
  }
  // B shard i is h x F_i: K-major over F_i, rows h, batch t
  DM_TRY(map_k(mapB, B, P.Fi, P.h, P.t, P.Fi, P.h * P.Fi, dm::kBBoxRows));
  return DOMINO_OK;
}

// Buffers and maps of one backward pass that do not change across row chunks.
struct BwdCtx {
  uint16_t* dZ;
  uint16_t* Hb;
  float* parts;
  CUtensorMap mapBmn, mapAmn, mapDZk, mapDZmn, mapHmn;
};

domino_status bwd_ctx(const Plan& P, const uint16_t* A, const uint16_t* B, uint8_t* ws, BwdCtx* C) {
  C->dZ = reinterpret_cast<uint16_t*>(ws + P.off_dz);
  C->Hb = reinterpret_cast<uint16_t*>(ws + P.off_hb);
  C->parts = reinterpret_cast<float*>(ws + P.off_part);
  // weight maps: B_i (h x F_i) read MN-major (N = F_i, K = h); A_i (R_i x h) read MN-major (N = h, K = R_i)
  DM_TRY(map_mn(&C->mapBmn, B, P.Fi, P.h, P.t, P.Fi, P.h * P.Fi));
  DM_TRY(map_mn(&C->mapAmn, A, P.h, P.Ri, P.t, P.h, P.Ri * P.h));
  DM_TRY(map_k(&C->mapDZk, C->dZ, P.Ri, P.m, P.t, P.a_rows, P.Ri, 128));
  DM_TRY(map_mn(&C->mapDZmn, C->dZ, P.Ri, P.m, P.t, P.a_rows, P.Ri));
  DM_TRY(map_mn(&C->mapHmn, C->Hb, P.Fi, P.m, P.t, P.F, P.Fi));
  return DOMINO_OK;
}

// Backward of one MLP for the row chunk starting at X_c / gY_c / gX_c (m rows): dH with the
// activation backward -> dZ, H; gB += gY_c^T H; per column chunk the gX partials (compute stream)
// and their shard-sum into gX_c (reduction stream); gA += dZ^T X_c, overlapping that reduction.
domino_status mlp_chunk_bwd(domino_handle H, const Plan& P, const Streams& S, SlotRing& R, const BwdCtx& C,
                            const uint16_t* X_c, const uint16_t* save_c, const uint16_t* gY_c, uint16_t* gX_c,
                            float* gA, float* gB) {
  CUtensorMap mapGYk, mapGYmn, mapXmn;
  DM_TRY(map_k(&mapGYk, gY_c, P.h, P.m, 1, P.h, 0, 128));
  DM_TRY(map_mn(&mapGYmn, gY_c, P.h, P.m, 1, P.h, 0));
  DM_TRY(map_mn(&mapXmn, X_c, P.h, P.m, 1, P.h, 0));
  // dH_i = gY_c . B_i, with the activation backward in the epilogue -> dZ (dG|dU), H
  {
    const int variant = P.gated ? dm::GV_BWD_GLU : dm::GV_BWD_ACT;
    GemmArgs a = gemm_args(variant, P.t, P.m, P.Fi, P.h, 3);
    a.act = P.act;
    a.b_bmul = 1;
    a.cross_batch = 1;  // the shards share gY
    a.in0 = save_c;
    a.ldi = P.a_rows;
    a.bsi = P.Ri;
    a.offi = P.Fi;
    a.out0 = C.dZ;
    a.ld0 = P.a_rows;
    a.bs0 = P.Ri;
    a.off0 = P.Fi;
    a.out1 = C.Hb;
    a.ld1 = P.F;
    a.bs1 = P.Fi;
    // epilogue maps: saved Z (or G, U) of the chunk in, dZ (or dG, dU) and H out; each branch has
    // its own base so a column tail is clipped at F_i
    dm::EpiMaps em = {};
    DM_TRY(map_epi_bf16(&em.m[0], save_c, P.Fi, P.m, P.t, P.a_rows, P.Ri));
    DM_TRY(map_epi_bf16(&em.m[2], C.dZ, P.Fi, P.m, P.t, P.a_rows, P.Ri));
    if (P.gated) {
      DM_TRY(map_epi_bf16(&em.m[1], save_c + P.Fi, P.Fi, P.m, P.t, P.a_rows, P.Ri));
      DM_TRY(map_epi_bf16(&em.m[3], C.dZ + P.Fi, P.Fi, P.m, P.t, P.a_rows, P.Ri));
    }
    DM_TRY(map_epi_bf16(&em.m[4], C.Hb, P.Fi, P.m, P.t, P.F, P.Fi));
    DM_TRY(run_gemm(H, DOMINO_K_GEMM_DGRAD_H, variant, mapGYk, C.mapBmn, a, S.comp, &em));
  }
  // gB_i += gY_c^T . H_i   (D = h x F_i, K = tokens of the chunk)
  {
    GemmArgs a = gemm_args(dm::GV_WGRAD, P.t, P.h, P.Fi, P.m, 4);
    a.b_bmul = 1;
    a.cross_batch = 1;  // the shards share gY
    a.out0 = gB;
    a.ld0 = P.Fi;
    a.bs0 = P.h * P.Fi;
    DM_TRY(run_gemm(H, DOMINO_K_GEMM_WGRAD_B, dm::GV_WGRAD, mapGYmn, C.mapHmn, a, S.comp));
  }
  // gX partials: P_i = dZ_i . A_i (D = m x n per column chunk), reduced on the reduction stream
  for (int qc = 0; qc < P.q; ++qc) {
    if (P.sched == DOMINO_SCHED_FUSED) {
      GemmArgs a = gemm_args(dm::GV_BWD_REDUCE, P.t, P.m, P.n, P.Ri, 5);
      a.a_bmul = 1;
      a.b_row_off = int32_t(qc * P.n);
      a.b_bmul = 1;
      DM_TRY(run_fused_reduce(H, DOMINO_K_GEMM_DGRAD_X, dm::GV_BWD_REDUCE, C.mapDZk, C.mapAmn, a, nullptr,
                              gX_c + qc * P.n, P.h, C.parts, P.part_slot, S.comp));
      continue;
    }
    int slot;
    DM_TRY(slot_acquire(H, P, S, R, &slot));
    float* part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(C.parts) + P.part_slot * slot);
    GemmArgs a = gemm_args(dm::GV_BWD_PARTIAL, P.t, P.m, P.n, P.Ri, 5);
    a.a_bmul = 1;
    a.b_row_off = int32_t(qc * P.n);
    a.b_bmul = 1;
    a.out0 = part;
    a.ld0 = P.n;
    a.bs0 = P.m * P.n;
    dm::EpiMaps em = {};
    DM_TRY(map_f32_out(&em.m[0], part, P.n, P.m, P.t));
    DM_TRY(run_gemm(H, DOMINO_K_GEMM_DGRAD_X, dm::GV_BWD_PARTIAL, C.mapDZk, C.mapAmn, a, S.comp, &em));
    DM_TRY(slot_handoff(H, S, slot));
    DM_TRY(run_shard_sum(H, part, P.t, P.m, P.n, nullptr, 0, gX_c + qc * P.n, P.h, P.reduce_ctas, S.red));
    DM_TRY(slot_release(H, S, R, slot));
  }
  // gA_i += dZ_i^T . X_c (D = R_i x h, K = tokens), overlapping the gX reduction
  {
    GemmArgs a = gemm_args(dm::GV_WGRAD, P.t, P.Ri, P.h, P.m, 6);
    a.a_bmul = 1;
    a.out0 = gA;
    a.ld0 = P.h;
    a.bs0 = P.Ri * P.h;
    DM_TRY(run_gemm(H, DOMINO_K_GEMM_WGRAD_A, dm::GV_WGRAD, C.mapDZmn, mapXmn, a, S.comp));
  }
  return DOMINO_OK;
}

domino_status ensure_row_events(domino_handle H, int p) {
  while (int(H->ev_row.size()) < p) {
    cudaEvent_t e;
    DM_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "cudaEventCreate");
    H->ev_row.push_back(e);
  }
  return DOMINO_OK;
}

// Before row chunk pc of a layer (other than the first processed): INTER waits only for the same
// row chunk of the previous layer; INTRA, at the layer's first chunk, for every row chunk of it.
domino_status wait_previous_layer(domino_handle H, const Plan& P, const Streams& S, int pc, bool first_chunk) {
  if (!S.overlap) return DOMINO_OK;
  if (P.sched == DOMINO_SCHED_INTER) {
    DM_CUDA(cudaStreamWaitEvent(S.comp, H->ev_row[pc], 0), "cudaStreamWaitEvent(row)");
  } else if (first_chunk) {
    for (int j = 0; j < P.p; ++j) DM_CUDA(cudaStreamWaitEvent(S.comp, H->ev_row[j], 0), "cudaStreamWaitEvent(row)");
  }
  return DOMINO_OK;
}

// Forward of the pre-LN residual stack; with `save` it also keeps, per layer, the LayerNorm output,
// the first-linear output and 1/sqrt(var + eps) for domino_stack_bwd.
domino_status stack_fwd_impl(domino_handle H, const Plan& P, const uint16_t* Z_in, const uint16_t* A,
                             const uint16_t* B, uint16_t* Z_out, uint8_t* save, void* ws, cudaStream_t caller) {
  DM_TRY(ensure_row_events(H, P.p));
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* Hbuf = reinterpret_cast<uint16_t*>(w + P.off_h);
  uint16_t* lnbuf = reinterpret_cast<uint16_t*>(w + P.off_ln);
  float* parts = reinterpret_cast<float*>(w + P.off_part);
  Streams S;
  DM_TRY(fork(H, P, caller, &S));
  const domino_status st = [&]() -> domino_status {
    SlotRing R;
    const int64_t a_layer = P.a_rows * P.h, b_layer = P.h * P.F;
    for (int l = 0; l < P.layers; ++l) {
      CUtensorMap mapA, mapB;
      DM_TRY(weight_maps_fwd(P, A + l * a_layer, B + l * b_layer, &mapA, &mapB));
      const uint16_t* src = (l == 0) ? Z_in : Z_out;
      uint8_t* sl = save ? save + l * P.save_layer : nullptr;
      for (int pc = 0; pc < P.p; ++pc) {
        NvtxChunk chunk_range_(pc);
        const int64_t r0 = pc * P.m;
        if (l > 0) DM_TRY(wait_previous_layer(H, P, S, pc, pc == 0));
        uint16_t* n_c = sl ? reinterpret_cast<uint16_t*>(sl + P.save_n) + r0 * P.h : lnbuf;
        float* rstd_c = sl ? reinterpret_cast<float*>(sl + P.save_rstd) + r0 : nullptr;
        uint16_t* act_c = sl ? reinterpret_cast<uint16_t*>(sl + P.save_act) + r0 * P.a_rows : nullptr;
        DM_TRY(launch(H, DOMINO_K_LAYERNORM, S.comp, "LayerNorm launch", [&] {
          return dm::launch_layernorm(src + r0 * P.h, P.m, P.h, P.eps, n_c, rstd_c, S.comp);
        }));
        R.tail = l == P.layers - 1 && pc == P.p - 1;
        DM_TRY(mlp_chunk_fwd(H, P, S, R, n_c, mapA, mapB, Hbuf, parts, act_c, src + r0 * P.h, Z_out + r0 * P.h, 2));
        if (S.overlap) DM_CUDA(cudaEventRecord(H->ev_row[pc], S.red), "cudaEventRecord(row)");
      }
    }
    return DOMINO_OK;
  }();
  return finish(H, S, caller, st);
}

// ---- attention sublayer ----------------------------------------------------------------------

// Tensor maps of the attention kernel for one row chunk: QKV (head dim, 3 * heads slots, position,
// sequence) and O (head dim, heads, position, sequence), 128-byte swizzle.
domino_status attn_maps(const Plan& P, const uint16_t* QKV, const uint16_t* O, CUtensorMap* tq, CUtensorMap* to) {
  const uint64_t nseq = uint64_t(P.m / P.seq);
  std::string err;
  {
    const uint64_t dims[4] = {128, uint64_t(3 * P.heads), uint64_t(P.seq), nseq};
    const uint64_t strides[3] = {256, uint64_t(3 * P.h) * 2, uint64_t(P.seq) * uint64_t(3 * P.h) * 2};
    const uint32_t box[4] = {64, 1, 128, 1};
    if (!dm::make_map(tq, 2, QKV, 4, dims, strides, box, &err)) return fail(DOMINO_ERR_CUDA, err);
  }
  {
    const uint64_t dims[4] = {128, uint64_t(P.heads), uint64_t(P.seq), nseq};
    const uint64_t strides[3] = {256, uint64_t(P.h) * 2, uint64_t(P.seq) * uint64_t(P.h) * 2};
    const uint32_t box[4] = {64, 1, 32, 1};
    if (!dm::make_map(to, 2, O, 4, dims, strides, box, &err)) return fail(DOMINO_ERR_CUDA, err);
  }
  return DOMINO_OK;
}

// Weight maps of one attention sublayer: Wqkv (h, 3h) K-major; Wo shards (h/t, h, t) like B.
domino_status weight_maps_attn(const Plan& P, const uint16_t* Wqkv, const uint16_t* Wo, CUtensorMap* mapW,
                               CUtensorMap* mapO) {
  const int64_t Kc = P.h / P.t;
  DM_TRY(map_k(mapW, Wqkv, P.h, 3 * P.h, 1, P.h, 0, dm::kBBoxRows));
  DM_TRY(map_k(mapO, Wo, Kc, P.h, P.t, Kc, P.h * Kc, dm::kBBoxRows));
  return DOMINO_OK;
}

// Attention sublayer for one row chunk Xc (m rows = whole sequences): the fused projection
// QKV = Xc . Wqkv^T (every shard's query, key and value heads), causal attention per (query block,
// head, sequence) into O, then the row-parallel output projection with its shard-sum (+ residual)
// exactly as the MLP's second linear, with O_i (the shard's heads) in place of H_i.
domino_status attn_chunk_fwd(domino_handle H, const Plan& P, const Streams& S, SlotRing& R, const uint16_t* Xc,
                             const CUtensorMap& mapW, const CUtensorMap& mapWo, uint16_t* QKV, uint16_t* O,
                             float* parts, const uint16_t* res_c, uint16_t* Yc) {
  CUtensorMap mapX;
  DM_TRY(map_k(&mapX, Xc, P.h, P.m, 1, P.h, 0, 128));
  {
    GemmArgs a = gemm_args(dm::GV_FWD_ACT, 1, P.m, 3 * P.h, P.h, 7);
    a.act = DOMINO_ACT_NONE;
    a.cross_batch = 1;  // groups of 16 M-tiles, as for the MLP's first linear
    a.out0 = QKV;
    a.ld0 = 3 * P.h;
    dm::EpiMaps em = {};
    DM_TRY(map_epi_bf16(&em.m[0], QKV, 3 * P.h, P.m, 1, 3 * P.h, 0));
    DM_TRY(run_gemm(H, DOMINO_K_GEMM_QKV, dm::GV_FWD_ACT, mapX, mapW, a, S.comp, &em));
  }
  {
    CUtensorMap tq, to;
    DM_TRY(attn_maps(P, QKV, O, &tq, &to));
    dm::AttnArgs aa;
    aa.seq = P.seq;
    aa.heads = P.heads;
    aa.nhi = P.heads / P.t;
    aa.n_qblk = int32_t(cdiv(P.seq, 128));
    aa.scale_log2 = float(1.4426950408889634 / std::sqrt(128.0));
    aa.err_site = 8 << 4;
    DM_TRY(launch(H, DOMINO_K_ATTN, S.comp, "attention launch",
                  [&] { return dm::launch_attention(tq, to, aa, int(P.m / P.seq), P.attn_ctas, S.comp); }));
  }
  const int64_t Kc = P.h / P.t;
  CUtensorMap mapO;
  DM_TRY(map_k(&mapO, O, Kc, P.m, P.t, P.h, Kc, 128));
  return second_linear(H, P, S, R, DOMINO_K_GEMM_OPROJ, mapO, mapWo, Kc, parts, res_c, Yc, 9);
}

// Stack of pre-LN Transformer blocks: sublayers attention, MLP, attention, ... each over all row
// chunks, each chunk waiting (INTER) for the same chunk of the previous sublayer or (INTRA) for
// the whole previous sublayer before its LayerNorm.
domino_status block_fwd_impl(domino_handle H, const Plan& P, const uint16_t* Z_in, const uint16_t* Wqkv,
                             const uint16_t* Wo, const uint16_t* A, const uint16_t* B, uint16_t* Z_out, void* ws,
                             cudaStream_t caller) {
  DM_TRY(ensure_row_events(H, P.p));
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* QKV = reinterpret_cast<uint16_t*>(w + P.off_qkv);
  uint16_t* O = reinterpret_cast<uint16_t*>(w + P.off_o);
  uint16_t* lnbuf = reinterpret_cast<uint16_t*>(w + P.off_ln);
  uint16_t* Hbuf = reinterpret_cast<uint16_t*>(w + P.off_h);
  float* parts = reinterpret_cast<float*>(w + P.off_part);
  Streams S;
  DM_TRY(fork(H, P, caller, &S));
  const domino_status st = [&]() -> domino_status {
    SlotRing R;
    const int64_t qkv_layer = 3 * P.h * P.h, o_layer = P.h * P.h;
    const int64_t a_layer = P.a_rows * P.h, b_layer = P.h * P.F;
    for (int l = 0; l < P.layers; ++l) {
      CUtensorMap mapW, mapWo, mapA, mapB;
      DM_TRY(weight_maps_attn(P, Wqkv + l * qkv_layer, Wo + l * o_layer, &mapW, &mapWo));
      DM_TRY(weight_maps_fwd(P, A + l * a_layer, B + l * b_layer, &mapA, &mapB));
      for (int sub = 0; sub < 2; ++sub) {
        const uint16_t* src = (l == 0 && sub == 0) ? Z_in : Z_out;
        for (int pc = 0; pc < P.p; ++pc) {
          NvtxChunk chunk_range_(pc);
          const int64_t r0 = pc * P.m;
          if (l > 0 || sub > 0) DM_TRY(wait_previous_layer(H, P, S, pc, pc == 0));
          DM_TRY(launch(H, DOMINO_K_LAYERNORM, S.comp, "LayerNorm launch", [&] {
            return dm::launch_layernorm(src + r0 * P.h, P.m, P.h, P.eps, lnbuf, nullptr, S.comp);
          }));
          R.tail = l == P.layers - 1 && sub == 1 && pc == P.p - 1;
          if (sub == 0)
            DM_TRY(attn_chunk_fwd(H, P, S, R, lnbuf, mapW, mapWo, QKV, O, parts, src + r0 * P.h, Z_out + r0 * P.h));
          else
            DM_TRY(mlp_chunk_fwd(H, P, S, R, lnbuf, mapA, mapB, Hbuf, parts, nullptr, src + r0 * P.h,
                                 Z_out + r0 * P.h, 2));
          if (S.overlap) DM_CUDA(cudaEventRecord(H->ev_row[pc], S.red), "cudaEventRecord(row)");
        }
      }
    }
    return DOMINO_OK;
  }();
  return finish(H, S, caller, st);
}

}  // namespace

namespace dm {
// Lets other translation units of the library report a message through domino_last_error().
void set_last_error(const std::string& msg) { t_last_error = msg; }
// The handle checks every entry point starts with (non-null, bound to the current device), for
// other translation units of the library.
domino_status check_handle(domino_handle H) { return ready(H); }
}  // namespace dm

// =============================================================================================

extern "C" {

const char* domino_status_string(domino_status s) {
  switch (s) {
    case DOMINO_OK: return "DOMINO_OK";
    case DOMINO_ERR_INVALID_ARG: return "DOMINO_ERR_INVALID_ARG";
    case DOMINO_ERR_UNSUPPORTED: return "DOMINO_ERR_UNSUPPORTED";
    case DOMINO_ERR_ALIGNMENT: return "DOMINO_ERR_ALIGNMENT";
    case DOMINO_ERR_WORKSPACE: return "DOMINO_ERR_WORKSPACE";
    case DOMINO_ERR_CUDA: return "DOMINO_ERR_CUDA";
    case DOMINO_ERR_TIMEOUT: return "DOMINO_ERR_TIMEOUT";
    case DOMINO_ERR_DEVICE: return "DOMINO_ERR_DEVICE";
  }
  return "DOMINO_ERR_UNKNOWN";
}

const char* domino_last_error(void) { return t_last_error.c_str(); }

domino_status domino_create(domino_handle* out) {
  if (!out) return fail(DOMINO_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  int dev = 0, major = 0, minor = 0, sms = 0;
  DM_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  DM_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev), "cudaDeviceGetAttribute");
  DM_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev), "cudaDeviceGetAttribute");
  DM_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3)
    return fail(DOMINO_ERR_DEVICE, "this build targets sm_103a; device is sm_" + std::to_string(major) +
                                       std::to_string(minor));
  std::string err;
  if (!dm::tma_encoder_ready(&err)) return fail(DOMINO_ERR_DEVICE, err);
  domino_handle H = new domino_handle_s();
  H->device = dev;
  H->num_sms = sms;
  cudaError_t e = cudaStreamCreateWithFlags(&H->s_comp, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&H->s_red, cudaStreamNonBlocking);
  cudaEvent_t* evs[] = {&H->ev_fork, &H->ev_join_c, &H->ev_join_r, &H->ev_part[0],
                        &H->ev_part[1], &H->ev_red[0], &H->ev_red[1]};
  for (cudaEvent_t* ev : evs)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    domino_destroy(H);
    return cuda_fail(e, "domino_create");
  }
  *out = H;
  return DOMINO_OK;
}

domino_status domino_destroy(domino_handle H) {
  if (!H) return DOMINO_OK;
  if (H->s_comp) cudaStreamSynchronize(H->s_comp);
  if (H->s_red) cudaStreamSynchronize(H->s_red);
  for (auto& t : H->timed) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  for (auto e : H->timing_pool) cudaEventDestroy(e);
  for (auto e : H->ev_row) cudaEventDestroy(e);
  cudaEvent_t evs[] = {H->ev_fork, H->ev_join_c, H->ev_join_r, H->ev_part[0],
                       H->ev_part[1], H->ev_red[0], H->ev_red[1]};
  for (cudaEvent_t e : evs)
    if (e) cudaEventDestroy(e);
  if (H->s_comp) cudaStreamDestroy(H->s_comp);
  if (H->s_red) cudaStreamDestroy(H->s_red);
  delete H;
  return DOMINO_OK;
}

domino_status domino_workspace_size(const domino_cfg* cfg, int32_t pass, size_t* bytes) {
  if (!bytes) return fail(DOMINO_ERR_INVALID_ARG, "bytes is NULL");
  Plan P;
  DM_TRY(make_plan(cfg, pass, &P));
  *bytes = P.total;
  return DOMINO_OK;
}

domino_status domino_mlp_fwd(domino_handle H, const domino_cfg* cfg, const uint16_t* X,
                             const uint16_t* A, const uint16_t* B, uint16_t* Y, uint16_t* act_save,
                             void* ws, size_t ws_bytes, void* stream) {
  DM_TRY(ready(H));
  NvtxRange range_("domino_mlp_fwd");
  Plan P;
  DM_TRY(make_plan(cfg, DOMINO_PASS_FWD, &P));
  DM_TRY(check_ptr(X, "X"));
  DM_TRY(check_ptr(A, "A"));
  DM_TRY(check_ptr(B, "B"));
  DM_TRY(check_ptr(Y, "Y"));
  DM_TRY(check_ptr(act_save, "act_save", true));
  DM_TRY(check_ws(P, ws, ws_bytes));
  if (P.M == 0) return DOMINO_OK;
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  CUtensorMap mapA, mapB;
  DM_TRY(weight_maps_fwd(P, A, B, &mapA, &mapB));
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* Hbuf = reinterpret_cast<uint16_t*>(w + P.off_h);
  float* parts = reinterpret_cast<float*>(w + P.off_part);
  Streams S;
  DM_TRY(fork(H, P, caller, &S));
  const domino_status st = [&]() -> domino_status {
    SlotRing R;
    for (int pc = 0; pc < P.p; ++pc) {
      NvtxChunk chunk_range_(pc);
      const int64_t r0 = pc * P.m;
      R.tail = pc == P.p - 1;
      DM_TRY(mlp_chunk_fwd(H, P, S, R, X + r0 * P.h, mapA, mapB, Hbuf, parts,
                           act_save ? act_save + r0 * P.a_rows : nullptr, nullptr, Y + r0 * P.h, 1));
    }
    return DOMINO_OK;
  }();
  return finish(H, S, caller, st);
}

domino_status domino_stack_fwd(domino_handle H, const domino_cfg* cfg, const uint16_t* Z_in,
                               const uint16_t* A, const uint16_t* B, uint16_t* Z_out, void* ws,
                               size_t ws_bytes, void* stream) {
  DM_TRY(ready(H));
  NvtxRange range_("domino_stack_fwd");
  Plan P;
  DM_TRY(make_plan(cfg, DOMINO_PASS_STACK, &P));
  DM_TRY(check_ptr(Z_in, "Z_in"));
  DM_TRY(check_ptr(A, "A"));
  DM_TRY(check_ptr(B, "B"));
  DM_TRY(check_ptr(Z_out, "Z_out"));
  DM_TRY(check_ws(P, ws, ws_bytes));
  if (P.M == 0) return DOMINO_OK;
  return stack_fwd_impl(H, P, Z_in, A, B, Z_out, nullptr, ws, static_cast<cudaStream_t>(stream));
}

domino_status domino_stack_save_size(const domino_cfg* cfg, size_t* bytes) {
  if (!bytes) return fail(DOMINO_ERR_INVALID_ARG, "bytes is NULL");
  Plan P;
  DM_TRY(make_plan(cfg, DOMINO_PASS_STACK, &P));
  *bytes = P.M == 0 ? 0 : P.save_layer * size_t(P.layers);
  return DOMINO_OK;
}

domino_status domino_stack_fwd_train(domino_handle H, const domino_cfg* cfg, const uint16_t* Z_in,
                                     const uint16_t* A, const uint16_t* B, uint16_t* Z_out, void* save,
                                     size_t save_bytes, void* ws, size_t ws_bytes, void* stream) {
  DM_TRY(ready(H));
  NvtxRange range_("domino_stack_fwd_train");
  Plan P;
  DM_TRY(make_plan(cfg, DOMINO_PASS_STACK, &P));
  DM_TRY(check_ptr(Z_in, "Z_in"));
  DM_TRY(check_ptr(A, "A"));
  DM_TRY(check_ptr(B, "B"));
  DM_TRY(check_ptr(Z_out, "Z_out"));
  DM_TRY(check_ws(P, ws, ws_bytes));
  if (P.M == 0) return DOMINO_OK;
  if (!save || (reinterpret_cast<uintptr_t>(save) & 255u) != 0)
    return fail(DOMINO_ERR_INVALID_ARG, "save must be a 256-byte aligned device buffer");
  if (save_bytes < P.save_layer * size_t(P.layers))
    return fail(DOMINO_ERR_INVALID_ARG, "save buffer too small: need " +
                                            std::to_string(P.save_layer * size_t(P.layers)) + " bytes");
  return stack_fwd_impl(H, P, Z_in, A, B, Z_out, static_cast<uint8_t*>(save), ws, static_cast<cudaStream_t>(stream));
}

domino_status domino_stack_bwd(domino_handle H, const domino_cfg* cfg, const uint16_t* A, const uint16_t* B,
                               const void* save, size_t save_bytes, const uint16_t* gZ_out, uint16_t* gZ_in,
                               float* gA, float* gB, void* ws, size_t ws_bytes, void* stream) {
  DM_TRY(ready(H));
  NvtxRange range_("domino_stack_bwd");
  Plan P;
  DM_TRY(make_plan(cfg, DOMINO_PASS_STACK_BWD, &P));
  DM_TRY(check_ptr(A, "A"));
  DM_TRY(check_ptr(B, "B"));
  DM_TRY(check_ptr(gZ_out, "gZ_out"));
  DM_TRY(check_ptr(gZ_in, "gZ_in"));
  DM_TRY(check_ptr(gA, "gA"));
  DM_TRY(check_ptr(gB, "gB"));
  DM_TRY(check_ws(P, ws, ws_bytes));
  if (P.M == 0) return DOMINO_OK;
  if (!save || (reinterpret_cast<uintptr_t>(save) & 255u) != 0)
    return fail(DOMINO_ERR_INVALID_ARG, "save must be a 256-byte aligned device buffer");
  if (save_bytes < P.save_layer * size_t(P.layers))
    return fail(DOMINO_ERR_INVALID_ARG, "save buffer too small");
  DM_TRY(ensure_row_events(H, P.p));
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* gn = reinterpret_cast<uint16_t*>(w + P.off_gn);
  const uint8_t* sv = static_cast<const uint8_t*>(save);
  Streams S;
  DM_TRY(fork(H, P, caller, &S));
  const domino_status st = [&]() -> domino_status {
    SlotRing R;
    const int64_t a_layer = P.a_rows * P.h, b_layer = P.h * P.F;
    for (int l = P.layers - 1; l >= 0; --l) {
      BwdCtx C;
      DM_TRY(bwd_ctx(P, A + l * a_layer, B + l * b_layer, w, &C));
      const uint8_t* sl = sv + l * P.save_layer;
      const uint16_t* n_l = reinterpret_cast<const uint16_t*>(sl + P.save_n);
      const uint16_t* act_l = reinterpret_cast<const uint16_t*>(sl + P.save_act);
      const float* rstd_l = reinterpret_cast<const float*>(sl + P.save_rstd);
      // the gradient arriving at this layer's output: the caller's for the last layer, then the
      // running gradient kept in gZ_in
      const uint16_t* g = (l == P.layers - 1) ? gZ_out : gZ_in;
      for (int pc = P.p - 1; pc >= 0; --pc) {
        NvtxChunk chunk_range_(pc);
        const int64_t r0 = pc * P.m;
        if (l < P.layers - 1) DM_TRY(wait_previous_layer(H, P, S, pc, pc == P.p - 1));
        DM_TRY(mlp_chunk_bwd(H, P, S, R, C, n_l + r0 * P.h, act_l + r0 * P.a_rows, g + r0 * P.h, gn + r0 * P.h,
                             gA + l * a_layer, gB + l * b_layer));
        // LayerNorm backward plus the residual path for the chunk's rows, after its reductions
        DM_TRY(launch(H, DOMINO_K_LN_BWD, S.red, "LayerNorm backward launch", [&] {
          return dm::launch_layernorm_bwd(gn + r0 * P.h, n_l + r0 * P.h, rstd_l + r0, g + r0 * P.h,
                                          gZ_in + r0 * P.h, P.m, P.h, S.red);
        }));
        if (S.overlap) DM_CUDA(cudaEventRecord(H->ev_row[pc], S.red), "cudaEventRecord(row)");
      }
    }
    return DOMINO_OK;
  }();
  return finish(H, S, caller, st);
}

domino_status domino_mlp_bwd(domino_handle H, const domino_cfg* cfg, const uint16_t* X,
                             const uint16_t* A, const uint16_t* B, const uint16_t* act_save,
                             const uint16_t* gY, uint16_t* gX, float* gA, float* gB, void* ws,
                             size_t ws_bytes, void* stream) {
  DM_TRY(ready(H));
  NvtxRange range_("domino_mlp_bwd");
  Plan P;
  DM_TRY(make_plan(cfg, DOMINO_PASS_BWD, &P));
  DM_TRY(check_ptr(X, "X"));
  DM_TRY(check_ptr(A, "A"));
  DM_TRY(check_ptr(B, "B"));
  DM_TRY(check_ptr(act_save, "act_save"));
  DM_TRY(check_ptr(gY, "gY"));
  DM_TRY(check_ptr(gX, "gX"));
  DM_TRY(check_ptr(gA, "gA"));
  DM_TRY(check_ptr(gB, "gB"));
  DM_TRY(check_ws(P, ws, ws_bytes));
  if (P.M == 0) return DOMINO_OK;
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  BwdCtx C;
  DM_TRY(bwd_ctx(P, A, B, static_cast<uint8_t*>(ws), &C));
  Streams S;
  DM_TRY(fork(H, P, caller, &S));
  const domino_status st = [&]() -> domino_status {
    SlotRing R;
    // row chunks in reverse order, as the backward pass runs the forward schedule backwards
    for (int pc = P.p - 1; pc >= 0; --pc) {
      NvtxChunk chunk_range_(pc);
      const int64_t r0 = pc * P.m;
      DM_TRY(mlp_chunk_bwd(H, P, S, R, C, X + r0 * P.h, act_save + r0 * P.a_rows, gY + r0 * P.h, gX + r0 * P.h,
                           gA, gB));
    }
    return DOMINO_OK;
  }();
  return finish(H, S, caller, st);
}

domino_status domino_mlp_fwd_fp8(domino_handle H, const domino_cfg* cfg, const uint8_t* X8, const uint8_t* A8,
                                 const uint8_t* B8, const float* scales, uint16_t* Y, void* ws, size_t ws_bytes,
                                 void* stream) {
  DM_TRY(ready(H));
  NvtxRange range_("domino_mlp_fwd_fp8");
  Plan P;
  DM_TRY(make_plan(cfg, DOMINO_PASS_FWD_FP8, &P));
  DM_TRY(check_ptr(X8, "X8"));
  DM_TRY(check_ptr(A8, "A8"));
  DM_TRY(check_ptr(B8, "B8"));
  DM_TRY(check_ptr(Y, "Y"));
  if (!scales) return fail(DOMINO_ERR_INVALID_ARG, "scales is NULL");
  for (int i = 0; i < 4; ++i)
    if (!(scales[i] > 0.0f) || !std::isfinite(scales[i]))
      return fail(DOMINO_ERR_INVALID_ARG, "scales must be finite and > 0");
  DM_TRY(check_ws(P, ws, ws_bytes));
  if (P.M == 0) return DOMINO_OK;
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  CUtensorMap mapA, mapB;
  DM_TRY(weight_maps_fp8(P, A8, B8, &mapA, &mapB));
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint8_t* H8 = w + P.off_h;
  float* parts = reinterpret_cast<float*>(w + P.off_part);
  const float sc[4] = {scales[0], scales[1], scales[2], scales[3]};
  Streams S;
  DM_TRY(fork(H, P, caller, &S));
  const domino_status st = [&]() -> domino_status {
    SlotRing R;
    for (int pc = 0; pc < P.p; ++pc) {
      NvtxChunk chunk_range_(pc);
      const int64_t r0 = pc * P.m;
      R.tail = pc == P.p - 1;
      DM_TRY(mlp_chunk_fwd_fp8(H, P, S, R, X8 + r0 * P.h, mapA, mapB, H8, parts, Y + r0 * P.h, sc));
    }
    return DOMINO_OK;
  }();
  return finish(H, S, caller, st);
}

domino_status domino_attn_fwd(domino_handle H, const domino_cfg* cfg, const uint16_t* X, const uint16_t* Wqkv,
                              const uint16_t* Wo, uint16_t* Y, void* ws, size_t ws_bytes, void* stream) {
  DM_TRY(ready(H));
  NvtxRange range_("domino_attn_fwd");
  Plan P;
  DM_TRY(make_plan(cfg, DOMINO_PASS_ATTN, &P));
  DM_TRY(check_ptr(X, "X"));
  DM_TRY(check_ptr(Wqkv, "Wqkv"));
  DM_TRY(check_ptr(Wo, "Wo"));
  DM_TRY(check_ptr(Y, "Y"));
  DM_TRY(check_ws(P, ws, ws_bytes));
  if (P.M == 0) return DOMINO_OK;
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  CUtensorMap mapW, mapWo;
  DM_TRY(weight_maps_attn(P, Wqkv, Wo, &mapW, &mapWo));
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* QKV = reinterpret_cast<uint16_t*>(w + P.off_qkv);
  uint16_t* O = reinterpret_cast<uint16_t*>(w + P.off_o);
  float* parts = reinterpret_cast<float*>(w + P.off_part);
  Streams S;
  DM_TRY(fork(H, P, caller, &S));
  const domino_status st = [&]() -> domino_status {
    SlotRing R;
    for (int pc = 0; pc < P.p; ++pc) {
      NvtxChunk chunk_range_(pc);
      const int64_t r0 = pc * P.m;
      R.tail = pc == P.p - 1;
      DM_TRY(attn_chunk_fwd(H, P, S, R, X + r0 * P.h, mapW, mapWo, QKV, O, parts, nullptr, Y + r0 * P.h));
    }
    return DOMINO_OK;
  }();
  return finish(H, S, caller, st);
}

domino_status domino_block_fwd(domino_handle H, const domino_cfg* cfg, const uint16_t* Z_in, const uint16_t* Wqkv,
                               const uint16_t* Wo, const uint16_t* A, const uint16_t* B, uint16_t* Z_out, void* ws,
                               size_t ws_bytes, void* stream) {
  DM_TRY(ready(H));
  NvtxRange range_("domino_block_fwd");
  Plan P;
  DM_TRY(make_plan(cfg, DOMINO_PASS_BLOCK, &P));
  DM_TRY(check_ptr(Z_in, "Z_in"));
  DM_TRY(check_ptr(Wqkv, "Wqkv"));
  DM_TRY(check_ptr(Wo, "Wo"));
  DM_TRY(check_ptr(A, "A"));
  DM_TRY(check_ptr(B, "B"));
  DM_TRY(check_ptr(Z_out, "Z_out"));
  if (Z_out == Z_in) return fail(DOMINO_ERR_INVALID_ARG, "Z_out may not alias Z_in");
  DM_TRY(check_ws(P, ws, ws_bytes));
  if (P.M == 0) return DOMINO_OK;
  return block_fwd_impl(H, P, Z_in, Wqkv, Wo, A, B, Z_out, ws, static_cast<cudaStream_t>(stream));
}

domino_status domino_shard_sum(const float* Pp, int32_t t, int64_t rows, int64_t cols,
                               const uint16_t* residual, int64_t ld_res, uint16_t* Y, int64_t ld_y,
                               void* stream) {
  if (t < 1 || rows < 0 || cols < 0) return fail(DOMINO_ERR_INVALID_ARG, "need t >= 1, rows, cols >= 0");
  if (cols % 8 != 0) return fail(DOMINO_ERR_ALIGNMENT, "cols must be a multiple of 8");
  // the kernel's grid-stride loop counts 16-byte vectors in 32 bits: below 2^31 it cannot wrap
  if (rows * (cols / 8) >= (int64_t(1) << 31)) return fail(DOMINO_ERR_UNSUPPORTED, "too many elements");
  if (ld_y < cols || (ld_y % 8) != 0) return fail(DOMINO_ERR_ALIGNMENT, "ld_y must be >= cols and a multiple of 8");
  if (residual && (ld_res < cols || (ld_res % 8) != 0))
    return fail(DOMINO_ERR_ALIGNMENT, "ld_res must be >= cols and a multiple of 8");
  if (rows == 0 || cols == 0) return DOMINO_OK;
  DM_TRY(check_ptr(Pp, "P"));
  DM_TRY(check_ptr(Y, "Y"));
  DM_TRY(check_ptr(residual, "residual", true));
  int dev = 0, sms = 0;
  DM_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  DM_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute");
  DM_CUDA(dm::launch_shard_sum(Pp, t, rows, cols, residual, ld_res, Y, ld_y, sms * 4,
                               static_cast<cudaStream_t>(stream)),
          "shard-sum launch");
  return DOMINO_OK;
}

domino_status domino_act_eval(int32_t act, const float* a, const float* b, float* out, float* da, float* db,
                              int64_t n, void* stream) {
  if (act < DOMINO_ACT_NONE || act > DOMINO_ACT_BILINEAR) return fail(DOMINO_ERR_INVALID_ARG, "unknown activation");
  if (n < 0) return fail(DOMINO_ERR_INVALID_ARG, "n must be >= 0");
  if (n == 0) return DOMINO_OK;
  const bool g = gated(act);
  if (!a || !out || !da || (g && (!b || !db))) return fail(DOMINO_ERR_INVALID_ARG, "NULL vector");
  DM_CUDA(dm::launch_act_eval(act, a, b, out, da, db, n, static_cast<cudaStream_t>(stream)), "activation launch");
  return DOMINO_OK;
}

domino_status domino_device_status(domino_handle H, domino_status* out, int32_t* site) {
  DM_TRY(ready(H));
  if (!out) return fail(DOMINO_ERR_INVALID_ARG, "out is NULL");
  DM_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  int c1 = 0, c2 = 0, c3 = 0, c4 = 0;
  DM_CUDA(dm::take_gemm_fwd_error(&c1), "reading the device error word");
  DM_CUDA(dm::take_gemm_bwd_error(&c2), "reading the device error word");
  DM_CUDA(dm::take_attn_error(&c3), "reading the device error word");
  DM_CUDA(dm::take_gemm_fp8_error(&c4), "reading the device error word");
  const int code = c1 ? c1 : (c2 ? c2 : (c3 ? c3 : c4));
  *out = code ? DOMINO_ERR_TIMEOUT : DOMINO_OK;
  if (site) *site = code;
  return DOMINO_OK;
}

domino_status domino_timing_enable(domino_handle H, int32_t enable) {
  if (!H) return fail(DOMINO_ERR_INVALID_ARG, "handle is NULL");
  H->timing = enable != 0;
  return DOMINO_OK;
}

domino_status domino_timing_reset(domino_handle H) {
  if (!H) return fail(DOMINO_ERR_INVALID_ARG, "handle is NULL");
  for (auto& t : H->timed) {
    H->timing_pool.push_back(t.a);
    H->timing_pool.push_back(t.b);
  }
  H->timed.clear();
  return DOMINO_OK;
}

domino_status domino_timing_read(domino_handle H, int32_t kind, int64_t* launches, double* total_ms) {
  if (!H || !launches || !total_ms) return fail(DOMINO_ERR_INVALID_ARG, "NULL argument");
  if (kind < 0 || kind >= DOMINO_K_COUNT) return fail(DOMINO_ERR_INVALID_ARG, "bad kernel kind");
  int64_t n = 0;
  double ms = 0.0;
  for (auto& t : H->timed) {
    if (t.kind != kind) continue;
    DM_CUDA(cudaEventSynchronize(t.b), "cudaEventSynchronize");
    float f = 0.0f;
    DM_CUDA(cudaEventElapsedTime(&f, t.a, t.b), "cudaEventElapsedTime");
    ms += f;
    ++n;
  }
  *launches = n;
  *total_ms = ms;
  return DOMINO_OK;
}

domino_status domino_timing_trace(domino_handle H, int64_t capacity, int32_t* kinds, double* start_ms,
                                  double* end_ms, int64_t* count) {
  if (!H || !count) return fail(DOMINO_ERR_INVALID_ARG, "NULL argument");
  if (capacity < 0 || (capacity > 0 && (!kinds || !start_ms || !end_ms)))
    return fail(DOMINO_ERR_INVALID_ARG, "capacity must be >= 0 and the arrays non-NULL");
  *count = int64_t(H->timed.size());
  if (H->timed.empty()) return DOMINO_OK;
  const cudaEvent_t t0 = H->timed.front().a;
  const int64_t n = std::min<int64_t>(capacity, *count);
  for (int64_t i = 0; i < n; ++i) {
    const TimedLaunch& t = H->timed[size_t(i)];
    DM_CUDA(cudaEventSynchronize(t.b), "cudaEventSynchronize");
    float a = 0.0f, b = 0.0f;
    DM_CUDA(cudaEventElapsedTime(&a, t0, t.a), "cudaEventElapsedTime");
    DM_CUDA(cudaEventElapsedTime(&b, t0, t.b), "cudaEventElapsedTime");
    kinds[i] = t.kind;
    start_ms[i] = a;
    end_ms[i] = b;
  }
  return DOMINO_OK;
}

domino_status domino_debug_skip_reduce(domino_handle H, int32_t enable) {
  if (!H) return fail(DOMINO_ERR_INVALID_ARG, "handle is NULL");
  H->skip_reduce = enable != 0;
  return DOMINO_OK;
}

domino_status domino_selftest_wait_timeout(domino_handle H, uint32_t timeout_us, void* stream) {
  DM_TRY(ready(H));
  if (timeout_us < 1 || timeout_us > 1000000u)
    return fail(DOMINO_ERR_INVALID_ARG, "timeout_us must be in [1, 1000000]");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return launch(H, DOMINO_K_COUNT, st, "self-test launch", [&] {
    return dm::launch_wait_selftest(uint64_t(timeout_us) * 1000u, DOMINO_SELFTEST_SITE, st);
  });
}

domino_status domino_debug_fail_launch(domino_handle H, int32_t nth) {
  if (!H) return fail(DOMINO_ERR_INVALID_ARG, "handle is NULL");
  if (nth < 0) return fail(DOMINO_ERR_INVALID_ARG, "nth must be >= 0");
  H->fail_countdown = nth;
  return DOMINO_OK;
}

domino_status domino_launch_count(domino_handle H, int64_t* launches) {
  if (!H || !launches) return fail(DOMINO_ERR_INVALID_ARG, "NULL argument");
  *launches = H->launches;
  return DOMINO_OK;
}

}  // extern "C"
