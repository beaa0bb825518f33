/*
 * domino.h -- C ABI of the GB300 (sm_103a) chunked tensor-parallel MLP.
 *
 * The operation is the tensor-parallel Transformer MLP written as XAB=Y and followed by
 * AllReduce(Y) ("DeepSpeed-Domino 深度解析", section "TP 的数据依赖：通信为何难以隐藏"):
 *
 *     Y = sum_{i<t} act(X . A_i^T) . B_i^T
 *
 * with the first linear column-parallel (shard i owns output features of A) and the second
 * row-parallel (shard i produces a partial sum P_i that the AllReduce adds up), as in the
 * nxmr.cn DP/TP/PP article, §3.1 "TP的切分方式与计算模式".  On one GPU the t shards are
 * emulated in device memory: each shard's fp32 partial is written to its own buffer and an
 * on-device shard-sum kernel stands in for the AllReduce.  The work is split as Domino does
 * ("Domino 核心设计：三种张量切分策略"): p row chunks of X along the token (batch)
 * dimension, q column chunks of B along its last (output) dimension, or both (2D).  The
 * reduction of chunk k runs on a second CUDA stream while the GEMMs of chunk k+1 run.
 *
 * Conventions shared by every entry point:
 *  - All tensor arguments are DEVICE pointers owned by the caller.  bf16 tensors are passed
 *    as uint16_t bit patterns; fp32 tensors as float.  Layouts are row-major, nn.Linear
 *    [out, in] orientation:
 *        X, gX, gY, Y, Z : M x h
 *        A : t contiguous shards; shard i is F_i x h, or 2F_i x h for gated activations
 *            (F_i gate rows followed by F_i up rows).  F_i = ffn / t.
 *        B : t contiguous shards; shard i is h x F_i.
 *        gA, gB : fp32, same shapes as A and B.
 *  - Every pointer must be 16-byte aligned; h, F_i and h/q must be multiples of 8.
 *  - The library allocates no device memory at run time.  Scratch space is the caller's
 *    workspace, whose size domino_workspace_size() returns; it must be 256-byte aligned.  The
 *    one exception is the fixed 64 MiB scratch array of domino_mlp_fwd_noalloc, a static device
 *    array of the library's module: every device that loads the module holds it until the
 *    process exits (reserved when the module loads, at context creation under eager module
 *    loading, else on first use, which may be the first domino_mlp_fwd_noalloc call).
 *  - Calls are asynchronous with respect to the host: work is ordered after prior work on
 *    `stream` (a cudaStream_t; NULL is the legacy default stream) and, on return, every
 *    launch is enqueued and joined back into `stream`.  Inputs must stay valid and outputs
 *    untouched until `stream` reaches that point.
 *  - Arguments are validated before anything is launched; a failed validation returns an
 *    error and launches nothing.  No C++ exception crosses this boundary.
 *  - A handle is bound to the device current at domino_create() and is not thread-safe:
 *    use one handle per host thread (or serialise calls).
 *  - Device-side waits are bounded in time; a wait that expires makes the kernel record an
 *    error word and return early.  domino_device_status() reads and clears that word.
 */
#ifndef DOMINO_H
#define DOMINO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DOMINO_API __attribute__((visibility("default")))
#else
#define DOMINO_API
#endif

typedef enum {
  DOMINO_OK = 0,
  DOMINO_ERR_INVALID_ARG = 1, /* null pointer, bad size, divisibility violated */
  DOMINO_ERR_UNSUPPORTED = 2, /* valid request this build does not implement */
  DOMINO_ERR_ALIGNMENT = 3,   /* pointer or leading dimension not 16-byte aligned */
  DOMINO_ERR_WORKSPACE = 4,   /* workspace missing, misaligned or too small */
  DOMINO_ERR_CUDA = 5,        /* a CUDA runtime call failed; see domino_last_error() */
  DOMINO_ERR_TIMEOUT = 6,     /* a device-side wait expired (domino_device_status) */
  DOMINO_ERR_DEVICE = 7       /* current GPU is not sm_103 or lacks a needed driver entry */
} domino_status;

typedef enum {
  DOMINO_ACT_NONE = 0,
  DOMINO_ACT_RELU = 1,
  DOMINO_ACT_GELU = 2,     /* exact form: x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)) */
  DOMINO_ACT_SWIGLU = 3,   /* gated: silu(gate) * up, silu(g) = g / (1 + exp(-g)) */
  DOMINO_ACT_BILINEAR = 4  /* gated: gate * up */
} domino_act;

/* How chunks are pipelined ("Domino 核心设计" and "实现与优化", figure 9):
 *  SERIAL: every kernel on the caller's stream, no overlap (the naive TP order).
 *  INTRA : reduction of chunk k on a side stream, overlapping the GEMMs of chunk k+1.  The
 *          call's last chunk has no chunk k+1: its last column block is reduced inside its GEMM
 *          as in FUSED (same arithmetic and bits).
 *  INTER : as INTRA; in the layer stack, row chunk j of layer l+1 starts as soon as the
 *          reductions of row chunk j of layer l finish (no wait for the whole layer).
 *  FUSED : the reduction is overlapped at tile granularity inside the second linear (and the
 *          input-gradient GEMM of the backward), the one-GPU analogue of GEMM + reduce-scatter
 *          tile pipelining ("04 · TP/SP 的通信-计算 overlap 与工程优化" §3, userbuffers): one
 *          persistent kernel computes, per output tile, the t shard partials in shard order
 *          and adds each, as it leaves the tensor-core accumulator, into an fp32 running sum
 *          held in the epilogue threads' registers (P_0, then + P_1, ..., one rounding per
 *          add); after the last shard the sum (plus the residual) is rounded once to bf16.
 *          A last round of output tiles that would keep at most half the GPU busy is shared
 *          by several CTA pairs per tile, each computing a group of shards whose partials it
 *          writes to the workspace; the tile's first pair adds them all in shard order.  Same
 *          arithmetic and order as the other schedules; everything runs on the caller's
 *          stream; the workspace holds no partial slots, only those of that last round
 *          (256 KiB per shard of each of its tiles). */
typedef enum {
  DOMINO_SCHED_SERIAL = 0,
  DOMINO_SCHED_INTRA = 1,
  DOMINO_SCHED_INTER = 2,
  DOMINO_SCHED_FUSED = 3
} domino_sched;

typedef enum {
  DOMINO_PASS_FWD = 0,       /* domino_mlp_fwd */
  DOMINO_PASS_BWD = 1,       /* domino_mlp_bwd */
  DOMINO_PASS_STACK = 2,     /* domino_stack_fwd, domino_stack_fwd_train */
  DOMINO_PASS_STACK_BWD = 3, /* domino_stack_bwd */
  DOMINO_PASS_ATTN = 4,      /* domino_attn_fwd */
  DOMINO_PASS_BLOCK = 5,     /* domino_block_fwd */
  DOMINO_PASS_FWD_FP8 = 6    /* domino_mlp_fwd_fp8 */
} domino_pass;

typedef struct {
  int64_t M;      /* tokens (batch x sequence); M % p == 0 */
  int64_t h;      /* hidden size */
  int64_t ffn;    /* F: ffn width (per branch for gated activations); F % t == 0 */
  int32_t t;      /* weight shards (emulated tensor-parallel ranks), >= 1 */
  int32_t p;      /* row chunks of X (token dimension), >= 1 */
  int32_t q;      /* column chunks of B's output dimension h, >= 1; h % q == 0 */
  int32_t act;    /* domino_act */
  int32_t sched;  /* domino_sched */
  int32_t layers; /* domino_stack_fwd only: number of layers (>= 1) */
  float ln_eps;   /* domino_stack_fwd only: LayerNorm epsilon (> 0) */
  int32_t flags;  /* reserved, must be 0 */
  int32_t heads;  /* attention passes only: attention heads, h / heads == 128, heads % t == 0 */
  int32_t seq;    /* attention passes only: tokens per sequence; M % (p * seq) == 0 */
  int32_t reduce_ctas; /* CTAs of each shard-sum launch (the AllReduce stand-in), >= 0; 0 = 4 per
                          SM.  A small budget leaves more of the SMs to the GEMMs it overlaps
                          (schedules INTRA / INTER); results do not depend on it. */
  int32_t attn_ctas;   /* attention passes only: CTAs of each attention launch, >= 0; 0 = one per
                          SM (the kernel is persistent over its work units); results do not
                          depend on it. */
} domino_cfg;

typedef struct domino_handle_s* domino_handle;

/* Creates a handle on the current device: two internal streams (compute and reduction,
 * both non-blocking) and a pool of events.  Fails with DOMINO_ERR_DEVICE on a GPU other
 * than compute capability 10.3.  *out is set to NULL on failure. */
DOMINO_API domino_status domino_create(domino_handle* out);

/* Destroys the handle after synchronising its internal streams.  NULL is accepted. */
DOMINO_API domino_status domino_destroy(domino_handle handle);

/* Bytes of workspace that `pass` needs for `cfg` (0 is possible).  Host-only. */
DOMINO_API domino_status domino_workspace_size(const domino_cfg* cfg, int32_t pass, size_t* bytes);

/* Forward of one MLP: Y = sum_i act(X . A_i^T) . B_i^T, bf16 output rounded once from the
 * fp32 shard-sum (shard order 0..t-1).  act_save (nullable) receives what the backward
 * needs: the bf16 first-linear output, M x F for non-gated activations, or M x 2F laid out
 * per shard as [gate_i | up_i] (columns i*2F_i .. (i+1)*2F_i) for gated ones.
 * Row-split results are bit-identical to p = 1. */
DOMINO_API domino_status domino_mlp_fwd(domino_handle handle, const domino_cfg* cfg, const uint16_t* X,
                             const uint16_t* A, const uint16_t* B, uint16_t* Y, uint16_t* act_save,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Backward of one MLP ("实现与优化" figure 10; "04 · TP/SP 的通信-计算 overlap 与工程优化" §1):
 *   dH = gY . Bfull,  dZ = dH * act'(.)  (gated: dG, dU),
 *   gX = sum_i dZ_i . A_i            (bf16; the shard-sum is the dgrad AllReduce stand-in),
 *   gA += dZ^T . X,  gB += gY^T . H   (fp32 accumulate into caller-owned main_grad buffers).
 * act_save is the buffer domino_mlp_fwd filled for the same X, A, B.  The gX reduction of
 * each row chunk overlaps the gA weight-gradient GEMM on the compute stream. */
DOMINO_API domino_status domino_mlp_bwd(domino_handle handle, const domino_cfg* cfg, const uint16_t* X,
                             const uint16_t* A, const uint16_t* B, const uint16_t* act_save,
                             const uint16_t* gY, uint16_t* gX, float* gA, float* gB,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Forward of one MLP, exactly as domino_mlp_fwd, for callers that cannot allocate device memory
 * when they run the layer (a plugin inside a framework that owns the whole memory pool and gives
 * out no workspace, a serving loop that forbids allocations after warm-up, code that must avoid
 * the device-wide synchronisation cudaMalloc/cudaFree may cause).  Not part of the method on the
 * pages: it has no counterpart there.
 * The scratch comes from a fixed 64 MiB array compiled into the library, which every GPU that
 * loads the library holds until the process exits; nothing is allocated.  Problems whose
 * domino_workspace_size(cfg, DOMINO_PASS_FWD) exceeds 64 MiB are rejected with
 * DOMINO_ERR_WORKSPACE and nothing is launched.
 * Each call outside stream capture looks up the array's device address on the current device
 * (the first such call may load the module and so reserve the array); a call made while `stream`
 * is being captured reuses the address the last uncaptured call on that device found, so make one
 * call on each device before any stream capture, else it fails with DOMINO_ERR_CUDA.  The handle
 * and the problem are checked before anything touches the device.  All calls share the one array: calls
 * whose work overlaps on the GPU (other streams, other host threads, other handles on the same
 * device) race on it and must be serialised by the caller.  The array keeps the last call's
 * contents; the forward overwrites every scratch byte it reads, so nothing needs clearing. */
DOMINO_API domino_status domino_mlp_fwd_noalloc(domino_handle handle, const domino_cfg* cfg,
                                                const uint16_t* X, const uint16_t* A, const uint16_t* B,
                                                uint16_t* Y, uint16_t* act_save, void* stream);

/* Pre-LN residual stack of cfg->layers layers ("实现与优化": LayerNorm, GeMM + act + GeMM,
 * residual):  Z_{l+1} = bf16(Z_l + sum_i act(LN(Z_l) . A_{l,i}^T) . B_{l,i}^T).
 * LN has no affine parameters and eps = cfg->ln_eps; its output is rounded to bf16 before
 * the first GEMM; the residual is added in fp32 to the shard-sum before the one rounding.
 * A and B hold cfg->layers consecutive layer blocks.  Z_out may equal Z_in. */
DOMINO_API domino_status domino_stack_fwd(domino_handle handle, const domino_cfg* cfg, const uint16_t* Z_in,
                               const uint16_t* A, const uint16_t* B, uint16_t* Z_out,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Training forward of the layer stack: as domino_stack_fwd, and additionally keeps in `save` what
 * domino_stack_bwd needs, per layer: the bf16 LayerNorm output (M x h), the bf16 first-linear
 * output (M x F, or M x 2F gated, laid out as act_save of domino_mlp_fwd) and the fp32
 * 1/sqrt(var + eps) of every row.  `save` is a 256-byte aligned device buffer of at least
 * domino_stack_save_size() bytes. */
DOMINO_API domino_status domino_stack_save_size(const domino_cfg* cfg, size_t* bytes);
DOMINO_API domino_status domino_stack_fwd_train(domino_handle handle, const domino_cfg* cfg,
                                                const uint16_t* Z_in, const uint16_t* A, const uint16_t* B,
                                                uint16_t* Z_out, void* save, size_t save_bytes,
                                                void* workspace, size_t workspace_bytes, void* stream);

/* Backward of the layer stack ("实现与优化" figure 10: the forward schedule in reverse).  From the
 * gradient gZ_out of the stack output, per layer l = L-1 .. 0 and row chunk (in reverse):
 *   gN = MLP_l input gradient (domino_mlp_bwd with X = the saved LayerNorm output),
 *   g  = bf16( g + r (gN - mean(gN) - N mean(gN N)) )   (LayerNorm backward + residual),
 * with gA, gB (L consecutive layer blocks, fp32) accumulated with +=.  gZ_in (M x h) receives the
 * gradient of the stack input; it also holds the running gradient between layers.  Workspace:
 * domino_workspace_size(cfg, DOMINO_PASS_STACK_BWD).  With DOMINO_SCHED_INTER, row chunk j of layer
 * l-1 starts once row chunk j of layer l has finished its LayerNorm backward. */
DOMINO_API domino_status domino_stack_bwd(domino_handle handle, const domino_cfg* cfg, const uint16_t* A,
                                          const uint16_t* B, const void* save, size_t save_bytes,
                                          const uint16_t* gZ_out, uint16_t* gZ_in, float* gA, float* gB,
                                          void* workspace, size_t workspace_bytes, void* stream);

/* FP8 variant of domino_mlp_fwd ("04 · TP/SP 的通信-计算 overlap 与工程优化" §4: FP8 halves what
 * moves, the reduction accumulates in higher precision).  Operands are E4M3 codes (OCP FP8:
 * 4 exponent bits, bias 7, 3 mantissa bits, largest finite 448, no infinities) with per-tensor
 * scales, host array scales = {sx, sa, sb, sh}: the real operands are sx*X8, sa*A8, sb*B8.
 *   Z = sx sa (X8 . A8^T) in fp32;  H = act(Z) (gated: glu);  H8 = e4m3(H / sh) (nearest, ties to
 *   even, saturating at +-448) for the second linear;  partials P_i = sh sb (H8_i . B8_i^T) and
 *   their shard-sum in fp32;  Y = bf16(sum), rounded once.
 * Layouts as domino_mlp_fwd, one byte per element: X8 M x h, A8 the A shards, B8 the B shards.
 * Needs h and ffn / t to be multiples of 16 (16-byte rows).  Power-of-two scales make the scaling
 * exact.  Same chunking and schedules; workspace: domino_workspace_size(cfg, DOMINO_PASS_FWD_FP8). */
DOMINO_API domino_status domino_mlp_fwd_fp8(domino_handle handle, const domino_cfg* cfg, const uint8_t* X8,
                                            const uint8_t* A8, const uint8_t* B8, const float* scales, uint16_t* Y,
                                            void* workspace, size_t workspace_bytes, void* stream);

/* Attention sublayer of one Transformer block ("TP 的数据依赖：通信为何难以隐藏": for the attention
 * layer of XAB=Y, X is the input, A the multi-head attention and B a linear layer; the AllReduce
 * follows):
 *   Y = sum_i Attn_i(X) . Wo_i^T,   Attn_i = causal self-attention of shard i's heads,
 * heads split over the t shards (Megatron style), with the same chunking (p row chunks holding
 * whole sequences, q column chunks of the output projection), schedules and fp32 shard-sum as
 * domino_mlp_fwd; bf16 output rounded once.  Per head (d = h / heads = 128): q, k, v = X . W^T,
 * o = softmax(q k^T / sqrt(d) over positions <= the query's, within its sequence) v.
 *   X:    M x h bf16; token r is position r % seq of sequence r / seq.
 *   Wqkv: t shards of (3 h/t) x h, each [query heads; key heads; value heads] of the shard, d rows
 *         per head, nn.Linear [out, in] layout.
 *   Wo:   t shards of h x (h/t); column j*d + e of shard i multiplies element e of its head j.
 * cfg->heads and cfg->seq are required; cfg->ffn and cfg->act are ignored.  Unsupported head
 * dimensions return DOMINO_ERR_UNSUPPORTED.  Workspace: domino_workspace_size(cfg,
 * DOMINO_PASS_ATTN). */
DOMINO_API domino_status domino_attn_fwd(domino_handle handle, const domino_cfg* cfg, const uint16_t* X,
                                         const uint16_t* Wqkv, const uint16_t* Wo, uint16_t* Y, void* workspace,
                                         size_t workspace_bytes, void* stream);

/* Stack of cfg->layers pre-LN Transformer blocks ("实现与优化", figure 9: one self-attention layer
 * and one MLP layer per block, LayerNorm and residual between them):
 *   Z += Attn(LN(Z));  Z += MLP(LN(Z))
 * LayerNorm as in domino_stack_fwd; the attention sublayer as in domino_attn_fwd, the MLP as in
 * domino_mlp_fwd; each sublayer's residual is added in fp32 to its shard-sum before the one bf16
 * rounding.  Per-layer weights are consecutive blocks: Wqkv (3h x h), Wo (h x h as t shards), A
 * and B as in domino_stack_fwd.  The sublayers run in the order attention (all row chunks), MLP
 * (all row chunks), next layer; with INTER a row chunk of one sublayer starts as soon as the
 * reductions of the same row chunk of the previous sublayer are done (the fig-9 interleaving:
 * a chunk's reduction overlaps the next chunk's compute).  Z_in is not modified; Z_out may not
 * alias it.  Workspace: domino_workspace_size(cfg, DOMINO_PASS_BLOCK). */
DOMINO_API domino_status domino_block_fwd(domino_handle handle, const domino_cfg* cfg, const uint16_t* Z_in,
                                          const uint16_t* Wqkv, const uint16_t* Wo, const uint16_t* A,
                                          const uint16_t* B, uint16_t* Z_out, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* The reduction step alone (the AllReduce stand-in):
 *   Y[r, c] = bf16( (residual[r, c]) + (((P_0[r,c] + P_1[r,c]) + ...) + P_{t-1}[r,c]) )
 * P: t slices of rows x cols fp32, slice i at P + i*rows*cols, row stride cols.
 * residual (nullable) has row stride ld_res; Y has row stride ld_y (elements).
 * cols must be a multiple of 8. */
DOMINO_API domino_status domino_shard_sum(const float* P, int32_t t, int64_t rows, int64_t cols,
                               const uint16_t* residual, int64_t ld_res, uint16_t* Y,
                               int64_t ld_y, void* stream);

/* The activation functions exactly as the GEMM epilogues evaluate them, on n fp32 device values:
 * non-gated: out = act(a), da = act'(a), db (nullable) = 0 when the separate and the combined
 * derivative code paths agree; gated: out = glu(a, b), da = d out/d a, db = d out/d b (b, db
 * required).  GeLU uses Phi from erf by Abramowitz & Stegun 7.1.26 (|erf error| <= 1.5e-7). */
DOMINO_API domino_status domino_act_eval(int32_t act, const float* a, const float* b, float* out, float* da,
                                         float* db, int64_t n, void* stream);

/* Reads and clears the device error word of every kernel of this library.  *out is
 * DOMINO_OK or DOMINO_ERR_TIMEOUT; *site (nullable) receives the code of the wait that
 * expired.  Synchronises the device. */
DOMINO_API domino_status domino_device_status(domino_handle handle, domino_status* out, int32_t* site);

/* Per-kernel timing: when enabled, each launch is bracketed by CUDA events on the stream it
 * is launched on.  domino_timing_read() synchronises on those events and returns, for one
 * kernel kind, the number of launches and their summed duration since the last reset. */
typedef enum {
  DOMINO_K_GEMM_FWD1 = 0,   /* first linear + activation epilogue */
  DOMINO_K_GEMM_FWD2 = 1,   /* second linear -> fp32 shard partials (FUSED: + shard-sum) */
  DOMINO_K_SHARD_SUM = 2,   /* shard-sum (AllReduce stand-in) */
  DOMINO_K_LAYERNORM = 3,
  DOMINO_K_GEMM_DGRAD_H = 4,/* gY . Bfull with activation-backward epilogue */
  DOMINO_K_GEMM_WGRAD_B = 5,/* gB += gY^T . H */
  DOMINO_K_GEMM_DGRAD_X = 6,/* dZ_i . A_i -> fp32 shard partials of gX (FUSED: + shard-sum) */
  DOMINO_K_GEMM_WGRAD_A = 7,/* gA += dZ^T . X */
  DOMINO_K_LN_BWD = 8,      /* LayerNorm backward + residual (layer stack) */
  DOMINO_K_GEMM_QKV = 9,    /* fused query/key/value projection of the attention sublayer */
  DOMINO_K_ATTN = 10,       /* causal multi-head attention */
  DOMINO_K_GEMM_OPROJ = 11, /* attention output projection -> fp32 shard partials (FUSED: + shard-sum) */
  DOMINO_K_COUNT = 12
} domino_kernel_kind;
DOMINO_API domino_status domino_timing_enable(domino_handle handle, int32_t enable);
DOMINO_API domino_status domino_timing_reset(domino_handle handle);
DOMINO_API domino_status domino_timing_read(domino_handle handle, int32_t kind, int64_t* launches,
                                 double* total_ms);

/* Launch timeline of the timed launches since the last domino_timing_reset (timing enabled), in
 * issue order: for launch i its kernel kind and the times (ms) of its start and end events relative
 * to the start event of the first timed launch.  Each launch is bracketed by events on the stream
 * it was launched on, so the start event completes once that stream reached the launch (its event
 * waits satisfied); kernels of the two internal streams can then be seen running side by side (the
 * time in which a shard-sum runs with no GEMM beside it is the reduction left exposed, "实现与优化").
 * Writes min(capacity, count) entries; *count receives the number of timed launches.  Synchronises
 * on the events it reads. */
DOMINO_API domino_status domino_timing_trace(domino_handle handle, int64_t capacity, int32_t* kinds,
                                             double* start_ms, double* end_ms, int64_t* count);

/* Measurement hook for the exposed-reduction figure ("按行切分输入 X：可达 100% 的通信隐藏": how
 * much of the reduction the chunk pipeline hides): with enable != 0, calls through `handle` under
 * the stream schedules (SERIAL, INTRA, INTER) run the same schedule with every shard-sum (the
 * AllReduce stand-in) replaced by a kernel of the same grid that does no reduction -- in layer
 * stacks it copies the residual into the output, elsewhere it does nothing -- and the call's last
 * chunk, which INTRA / INTER reduce inside its GEMM, runs the plain fp32-partial GEMM instead.  The
 * step time without the reduction is then comparable with the normal one.  Outputs written by a
 * shard-sum (Y, gX, the layer outputs) are WRONG while it is on; FUSED calls fail with
 * DOMINO_ERR_UNSUPPORTED.  0 (the default) restores the normal path. */
DOMINO_API domino_status domino_debug_skip_reduce(domino_handle handle, int32_t enable);

/* Failure-path self-test: launches a one-CTA kernel whose mbarrier wait can never complete.
 * After timeout_us (1 .. 1,000,000 microseconds) the bounded wait gives up, records
 * DOMINO_ERR_TIMEOUT with site DOMINO_SELFTEST_SITE in the device error word and the kernel
 * returns; the GPU context stays usable.  Read the result with domino_device_status(). */
#define DOMINO_SELFTEST_SITE 0x7F0
DOMINO_API domino_status domino_selftest_wait_timeout(domino_handle handle, uint32_t timeout_us, void* stream);

/* Test hook: the nth launch attempt from now (1-based) through `handle` fails with
 * DOMINO_ERR_CUDA ("injected launch failure") instead of launching; 0 disables.  A call that
 * fails this way returns after joining its internal streams back into the caller's stream. */
DOMINO_API domino_status domino_debug_fail_launch(domino_handle handle, int32_t nth);

/* Number of kernels this library has launched through `handle` since creation. */
DOMINO_API domino_status domino_launch_count(domino_handle handle, int64_t* launches);

DOMINO_API const char* domino_status_string(domino_status status);

/* Message of the last failed call on the calling host thread ("" if none). */
DOMINO_API const char* domino_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* DOMINO_H */
