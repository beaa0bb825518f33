// gemm.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a with fused epilogues.
//
// A CTA pair (cluster of 2, one CTA per SM) loops over 256 x 256 output tiles (128 x 256 per CTA;
// the gated first linear: 256 x 128 outputs from 256 gate + up columns) with
// tcgen05.mma.cta_group::2.  Warp roles in each CTA:
//   warp 0 (one lane)  TMA producer: per K step, its 128 rows of A and its 128-row half of B
//                      (128 bytes of K: 64 bf16 or 128 E4M3 codes) into a 6-stage shared-memory
//                      ring (128-byte swizzle); both CTAs' copies complete on the leader's barrier.
//   warp 1             TMEM alloc/dealloc (pair-wide); lane 0 of the leader issues the MMAs into
//                      one of two TMEM accumulators (2 x 256 fp32 columns) and commits them,
//                      multicast to both CTAs, to the ring's "empty" and the accumulator's "full"
//                      barriers.
//   warps 2-5          epilogue: tcgen05.ld of the accumulator (each warp its 32-lane quarter, one
//                      row per thread), the variant's epilogue, then the accumulator is handed
//                      back so tile i+1's epilogue overlaps tile i+2's main loop.  The fused
//                      shard-sum has eight epilogue warps (2-9, two per quarter) that keep their
//                      rows' running sums over the shards in registers.
// Every wait is bounded (ptx.cuh); on expiry the CTA drains what it has in flight, frees TMEM
// and returns, leaving a code in the translation unit's error word.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <atomic>

#include "actfn.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dm {

// Device error word of the GEMM kernels of the including translation unit.
static __device__ int g_gemm_err;

constexpr bool is_act_bwd(int epi) { return epi == EPI_ACT_BWD || epi == EPI_GLU_BWD; }

// Shared-memory ring geometry.  PAIR: a CTA pair computes a 256 x 256 tile with
// tcgen05.mma.cta_group::2; each CTA stages its own 128 rows of A and its half (128 rows) of B,
// 32 KiB per stage, 6 stages (5 when the activation-backward epilogue needs its staging space).
// Single CTA: 128 x 256 tiles, 48 KiB stages, 4 stages.
template <bool PAIR, int EPI>
struct Ring {
  static constexpr int kBRows = PAIR ? 128 : 256;        // B rows staged by one CTA
  static constexpr int kABytes = kBM * kBK * 2;           // 16 KiB
  static constexpr int kBBytes = kBRows * kBK * 2;        // 16 or 32 KiB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = PAIR ? (is_act_bwd(EPI) ? 5 : 6) : (is_act_bwd(EPI) ? 3 : 4);
  static constexpr int kTileM = PAIR ? 2 * kBM : kBM;     // rows of D per tile
};
constexpr int kCtrlBytes = 1024;

// Four epilogue warps, one per TMEM lane quarter (32 rows), all accumulator columns; the fused
// shard-sum has eight, two per lane quarter with 128 columns each, whose threads keep their row's
// running sums in registers.  Block = TMA warp + MMA warp + epilogue warps.
template <int EPI>
constexpr int epi_warps() { return EPI == EPI_F32_REDUCE ? 8 : 4; }
// The activation backward and the non-gated bf16 forward activation add two helper warps
// (sub-partitions 2 and 3) that do the arithmetic of lane quarter 1 for its reader warp, which shares
// a sub-partition with the MMA issuer.  (The same split for the E4M3 GeLU epilogue sped up its kernel
// alone but not the step, where it runs beside the previous chunk's shard-sum; not used there.)
template <int EPI>
constexpr int helper_warps() { return (is_act_bwd(EPI) || EPI == EPI_ACT_BF16) ? 2 : 0; }
// Accumulator slots between the reader and the helpers (4 KiB each, see epilogue_acc_reader).
constexpr int kAccSlots = 2;
template <int EPI>
constexpr int block_threads() { return 64 + 32 * (epi_warps<EPI>() + helper_warps<EPI>()); }
// Threads a CTA is compiled for.  The fused shard-sum's ten warps put three on some sub-partitions,
// whose 16K registers then allow at most 168 a thread; compiling it as if for 384 threads keeps
// the compiler within that bound.
template <int EPI>
constexpr int bound_threads() { return EPI == EPI_F32_REDUCE ? 384 : block_threads<EPI>(); }
// Epilogues that move data with TMA stage it in shared memory, per epilogue warp:
//  fp32 partials: two 4 KiB buffers (32 rows x 32 fp32, 128-byte swizzle);
//  activation backward: per warp that does arithmetic (epilogue warps 2-4 and the two helpers; the
//  reader of quarter 1 needs none) 4 KiB of inputs (Z or G, U) and 6 KiB of outputs (dZ or dG, dU;
//  H), as 32 rows x 32 bf16 boxes with 64-byte swizzle, then the reader's two 4 KiB slots.
//  forward activation: up to three 2 KiB output boxes (H; saved Z, or G and U), 64-byte swizzle; the
//  non-gated form (two boxes) for warps 2-4 and its two helpers, then the reader's two slots.
constexpr int kActBwdWarpBytes = 10240;
constexpr int kFwdWarpBytes = 6144;    // gated forward: H, G, U boxes
constexpr int kFwdActWarpBytes = 4096; // non-gated forward: H, Z boxes
constexpr bool is_act_fwd(int epi) { return epi == EPI_ACT_BF16 || epi == EPI_GLU_BF16; }
constexpr bool is_act_f8(int epi) { return epi == EPI_ACT_F8 || epi == EPI_GLU_F8; }
constexpr bool is_gated_b(int epi) { return epi == EPI_GLU_BF16 || epi == EPI_GLU_F8; }
template <int EPI>
constexpr int staging_bytes() {
  return EPI == EPI_F32_STORE ? 4 * 2 * 4096
                              : (is_act_bwd(EPI) ? 5 * kActBwdWarpBytes + 2 * 4096
                                                 : (EPI == EPI_ACT_BF16 ? 5 * kFwdActWarpBytes + 2 * 4096
                                                                        : (is_act_fwd(EPI) ? 4 * kFwdWarpBytes : 0)));
}
template <bool PAIR, int EPI>
constexpr int smem_bytes() {
  return 1024 /* alignment slack */ + kCtrlBytes + Ring<PAIR, EPI>::kStages * Ring<PAIR, EPI>::kStageBytes +
         staging_bytes<EPI>();
}
constexpr int kTmemCols = 2 * kBN;
constexpr int kGroupM = 8;  // tiles are visited in groups of 8 M-tiles for L2 reuse of B tiles
// With cross_batch, groups of 16 M-tiles walk the N-tiles of every batch: an A operand shared by the
// batches (the first linear's X) is then read once per launch instead of once per batch.
constexpr int kGroupMCross = 16;
constexpr uint64_t kDrainTimeoutNs = 200000000ull;
// How long the leader's producer waits for its peer's count of issued stages: longer than any single
// bounded wait, so the peer has left its loop by then unless its GPU stopped making progress.
constexpr uint64_t kPeerCountTimeoutNs = 4000000000ull;
constexpr uint64_t kPeerCopyGraceNs = 100000ull;  // last resort when the peer's count never came

__device__ __forceinline__ void decode_tile(int tile, const GemmArgs& a, int& g, int& mt, int& nt) {
  if (a.cross_batch) {
    const int ncomb = a.batches * a.n_tiles;  // (batch, N-tile) pairs, batch-major
    const int span = kGroupMCross * ncomb;
    const int grp = tile / span;
    const int first_m = grp * kGroupMCross;
    const int gsize = min(a.m_tiles - first_m, kGroupMCross);
    const int in = tile - grp * span;
    mt = first_m + in % gsize;
    const int nb = in / gsize;
    g = nb / a.n_tiles;
    nt = nb - g * a.n_tiles;
    return;
  }
  const int per_batch = a.m_tiles * a.n_tiles;
  g = tile / per_batch;
  const int r = tile - g * per_batch;
  const int span = kGroupM * a.n_tiles;
  const int grp = r / span;
  const int first_m = grp * kGroupM;
  const int gsize = min(a.m_tiles - first_m, kGroupM);
  const int in = r - grp * span;
  mt = first_m + in % gsize;
  nt = in / gsize;
}

// Roles of a unit on an output tile of the fused shard-sum.
enum : int {
  FT_WHOLE = 0,   // all shards, sums in registers, writes Y
  FT_HEAD = 1,    // stores the partials of its shards [lo, hi), then adds all the tile's slots in
                  // shard order and writes Y
  FT_HELPER = 2,  // stores the partials of its shards [lo, hi) for the head
};
struct FusedTile {
  int mt, nt;  // output tile
  int lo, hi;  // shards this unit computes, in order
  int role;
  int slot0;   // the tile's partial slots: slot0 + g holds shard g (split tiles only)
};

// Output tile o (0, 1, ...) of a unit of the fused shard-sum.  Units take tiles unit, unit + units,
// ... of the (M, N) space while whole rounds remain.  With a.split = s > 1, each of the `rest` tiles
// of the last round is shared by s units: unit u < rest * s takes tile j = u / s, shards
// [i t / s, (i + 1) t / s) for i = u % s; i = 0 is the tile's head.  Every partial is computed exactly
// as in a whole tile (the same products over the same K steps), and the head adds them in shard order.
__device__ __forceinline__ bool fused_tile(int o, const GemmArgs& a, int unit, int units, FusedTile& f) {
  const int tiles = a.m_tiles * a.n_tiles, t = a.batches;
  const int full = tiles / units, rest = tiles - full * units;
  int ot;
  if (o < full || (o == full && a.split <= 1)) {
    ot = o * units + unit;
    f.lo = 0;
    f.hi = t;
    f.role = FT_WHOLE;
    f.slot0 = 0;
  } else {
    if (o > full || unit >= rest * a.split) return false;
    const int j = unit / a.split, i = unit - j * a.split;
    ot = full * units + j;
    f.lo = i * t / a.split;
    f.hi = (i + 1) * t / a.split;
    f.role = i == 0 ? FT_HEAD : FT_HELPER;
    f.slot0 = j * t;
  }
  if (ot >= tiles) return false;
  int g;
  decode_tile(ot, a, g, f.mt, f.nt);
  return true;
}

// Sub-tile s (0, 1, ...) of a unit's sequence.  Every variant but the fused shard-sum visits tiles
// unit, unit + units, ... of the (batch, M, N) tile space; the fused shard-sum visits its output
// tiles (fused_tile) and, for each, its shards in order.  False past the end of the sequence.
template <int EPI>
__device__ __forceinline__ bool tile_at(int s, const GemmArgs& a, int unit, int units, int& g, int& mt, int& nt) {
  if constexpr (EPI == EPI_F32_REDUCE) {
    const int t = a.batches, full = (a.m_tiles * a.n_tiles) / units;
    const int o = s < full * t ? s / t : full;
    FusedTile f;
    if (!fused_tile(o, a, unit, units, f)) return false;
    g = f.lo + (s - o * t);
    if (g >= f.hi) return false;
    mt = f.mt;
    nt = f.nt;
    return true;
  } else {
    const int tile = unit + s * units;
    if (tile >= a.batches * a.m_tiles * a.n_tiles) return false;
    decode_tile(tile, a, g, mt, nt);
    return true;
  }
}

// Number of sub-tiles in a unit's sequence (tile_at), in closed form: the MMA issuer needs only the
// count, and the integer divisions of the tile order, on its thread between two tiles, would keep the
// tensor core waiting.
template <int EPI>
__device__ __forceinline__ int unit_subtiles(const GemmArgs& a, int unit, int units) {
  if constexpr (EPI == EPI_F32_REDUCE) {
    const int t = a.batches, tiles = a.m_tiles * a.n_tiles;
    const int full = tiles / units, rest = tiles - full * units;
    if (a.split <= 1) return (full + (unit < rest ? 1 : 0)) * t;
    if (unit >= rest * a.split) return full * t;
    const int i = unit % a.split;
    return full * t + (i + 1) * t / a.split - i * t / a.split;
  } else {
    const int total = a.batches * a.m_tiles * a.n_tiles;
    return unit < total ? (total - 1 - unit) / units + 1 : 0;
  }
}

// Bounded wait that ignores the abort flag (used while draining after an abort).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kDrainTimeoutNs) return;
  }
}

// CTA-pair operand ring after the producers stopped: the leader CTA's producer makes sure every
// stage copy either CTA issued has landed before the pair leaves.  Both CTAs' copies of ring use j
// (stage j % S, phase parity (j / S) & 1) complete on the leader's full barrier, armed by the leader
// for both CTAs' bytes.  `own` and `peer` count the uses each producer issued.  A stage is reused
// only after its previous use was consumed, which needed both CTAs' bytes, so per stage only the
// last use below max(own, peer) can still be pending; for it, bytes that will never come are
// balanced first (issued by the leader only: the peer's share is marked done; by the peer only: the
// leader arrives expecting the peer's share), then the phase is awaited (bounded).
template <int S>
__device__ __forceinline__ void drain_pair_ring(uint32_t full_bar0, uint32_t own, uint32_t peer,
                                                uint32_t stage_bytes) {
  const uint32_t end = own > peer ? own : peer;
#pragma unroll 1
  for (uint32_t s = 0; s < static_cast<uint32_t>(S) && s < end; ++s) {
    const uint32_t j = s + (end - 1u - s) / S * S;  // last use of stage s below `end`
    const uint32_t bar = full_bar0 + 8u * s;
    const bool by_own = j < own, by_peer = j < peer;
    if (by_own && !by_peer)
      mbar_complete_tx(bar, stage_bytes);
    else if (!by_own && by_peer)
      mbar_arrive_expect_tx(bar, stage_bytes);
    mbar_wait_drain(bar, (j / S) & 1u);
  }
}

__device__ __forceinline__ void store8_bf16(uint16_t* p, const float* v) {
  uint4 w;
  w.x = pack_bf16x2(v[0], v[1]);
  w.y = pack_bf16x2(v[2], v[3]);
  w.z = pack_bf16x2(v[4], v[5]);
  w.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = w;
}

__device__ __forceinline__ void load8_bf16(const uint16_t* p, float* v) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16lo(w.x); v[1] = bf16hi(w.x);
  v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
  v[4] = bf16lo(w.z); v[5] = bf16hi(w.z);
  v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
}

// Epilogue of NC accumulator columns of one tile for the calling thread's row.  `tacc` addresses
// this warp's TMEM lane quarter at the first of those columns (for the gated forward: at the
// first gate column; the matching up columns sit 128 columns further).  Every lane executes the
// TMEM loads; only global accesses are masked.  Inputs of the next 32-column chunk are loaded
// before the current chunk's TMEM load is awaited.
template <int EPI, int NC>
__device__ __forceinline__ void epilogue_cols(const GemmArgs& a, uint32_t tacc, int g, int row, int col0) {
  const bool row_ok = row < a.M;
  const int64_t rowoff = static_cast<int64_t>(row);
  if constexpr (EPI == EPI_GLU_BF16) {
#pragma unroll 1
    for (int cc = 0; cc < NC; cc += 32) {
      uint32_t rg[32], ru[32];
      tmem_ld32(tacc + cc, rg);
      tmem_ld32(tacc + 128 + cc, ru);
      tmem_ld_wait();
      const int col = col0 + cc;
      if (!row_ok) continue;
      uint16_t* o0 = static_cast<uint16_t*>(a.out0) + g * a.bs0 + rowoff * a.ld0 + col;
      uint16_t* o1 = a.out1 ? static_cast<uint16_t*>(a.out1) + g * a.bs1 + rowoff * a.ld1 + col : nullptr;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        if (col + 8 * s >= a.N) break;
        float hv[8], gv[8], uv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          gv[e] = __uint_as_float(rg[8 * s + e]);
          uv[e] = __uint_as_float(ru[8 * s + e]);
          hv[e] = glu_fwd(a.act, gv[e], uv[e]);
        }
        store8_bf16(o0 + 8 * s, hv);
        if (o1) {
          store8_bf16(o1 + 8 * s, gv);
          store8_bf16(o1 + a.off1 + 8 * s, uv);
        }
      }
    }
  } else {
#pragma unroll 1
    for (int cc = 0; cc < NC; cc += 32) {
      uint32_t r[32];
      tmem_ld32(tacc + cc, r);
      tmem_ld_wait();
      const int col = col0 + cc;
      if (!row_ok || col >= a.N) continue;
      if constexpr (EPI == EPI_ACT_BF16) {
        uint16_t* o0 = static_cast<uint16_t*>(a.out0) + g * a.bs0 + rowoff * a.ld0 + col;
        uint16_t* o1 = a.out1 ? static_cast<uint16_t*>(a.out1) + g * a.bs1 + rowoff * a.ld1 + col : nullptr;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          if (col + 8 * s >= a.N) break;
          float v[8], z[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            z[e] = __uint_as_float(r[8 * s + e]);
            v[e] = act_fwd(a.act, z[e]);
          }
          store8_bf16(o0 + 8 * s, v);
          if (o1) store8_bf16(o1 + 8 * s, z);
        }
      } else {  // EPI_F32_STORE / EPI_F32_ACCUM
        float* o0 = static_cast<float*>(a.out0) + g * a.bs0 + rowoff * a.ld0 + col;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          if (col + 4 * s >= a.N) break;
          float4 v = make_float4(__uint_as_float(r[4 * s]), __uint_as_float(r[4 * s + 1]),
                                 __uint_as_float(r[4 * s + 2]), __uint_as_float(r[4 * s + 3]));
          float4* dst = reinterpret_cast<float4*>(o0 + 4 * s);
          if constexpr (EPI == EPI_F32_ACCUM) {
            const float4 old = *dst;
            v.x += old.x; v.y += old.y; v.z += old.z; v.w += old.w;
          }
          *dst = v;
        }
      }
    }
  }
}

// Arithmetic of one 32-column chunk of the activation-backward epilogue for the calling thread's row,
// with the activation fixed at compile time: from the accumulator dH (r, fp32) and the saved
// pre-activation (zi: Z or G, ui: U, bf16 pairs), dZ = dH act'(Z) (gated: dG, dU) and the
// recomputed H = act(Z), as bf16 pairs.  The caller picks the activation once per chunk, so the
// 32 independent evaluations form one branch-free block whose latency chains overlap.
template <bool kGlu, int ACT>
__device__ __forceinline__ void bwd_act_chunk(const uint32_t (&zi)[16], const uint32_t (&ui)[16],
                                              const uint32_t (&r)[32], uint32_t (&o1)[16], uint32_t (&o2)[16],
                                              uint32_t (&oh)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const uint32_t zw = zi[e >> 1];
    float d1a, d1b, d2a = 0.f, d2b = 0.f, ha, hb;
    const float z0 = bf16lo(zw), z1 = bf16hi(zw);
    const float g0 = __uint_as_float(r[e]), g1 = __uint_as_float(r[e + 1]);
    if constexpr (kGlu) {
      const uint32_t uw = ui[e >> 1];
      glu_bwd(ACT, z0, bf16lo(uw), g0, d1a, d2a, ha);
      glu_bwd(ACT, z1, bf16hi(uw), g1, d1b, d2b, hb);
    } else {
      float da, db;
      act_fwd_grad(ACT, z0, ha, da);
      act_fwd_grad(ACT, z1, hb, db);
      d1a = g0 * da;
      d1b = g1 * db;
    }
    o1[e >> 1] = pack_bf16x2(d1a, d1b);
    o2[e >> 1] = pack_bf16x2(d2a, d2b);
    oh[e >> 1] = pack_bf16x2(ha, hb);
  }
}

// Where a warp of the activation-backward epilogue takes the accumulator from: its TMEM lane quarter
// directly, or a shared-memory slot that the quarter's reader warp filled (epilogue_acc_reader).
enum : int { ACC_TMEM = 0, ACC_SLOT = 1 };

// The accumulator hand-off of one TMEM lane quarter: 4 KiB slots of 32 rows x 32 fp32 (one 32-column
// chunk), 128-byte rows with 16-byte piece j of row r at position j ^ (r % 8).  Chunk k of the unit's
// sequence (8 per tile) goes to slot k % kAccSlots, so the reader runs one chunk ahead of each helper.
constexpr uint32_t kAccSlotBytes = 4096;

// Reader warp of TMEM lane quarter 1, the quarter read by the warp that shares a sub-partition with
// the MMA-issuing warp: for every tile of the unit it copies the accumulator, 32 columns at a time,
// into the slots, where the helper warp of the chunk (even chunks: helper 0, odd: helper 1) takes it
// (epilogue_act_bwd_tma with ACC_SLOT, epilogue_fwd_helper, epilogue_f8_helper), and hands the
// accumulator back to the MMA issuer as soon as all its chunks are copied.
// The arithmetic of the quarter then runs on other sub-partitions: done by the warp beside the MMA
// issuer, it delayed the issue of the tensor-core instructions and slowed the main loop (measured).
// Slot barriers: full (the 32 lanes of the reader arrive) and empty (the 32 lanes of the helper
// arrive), so every lane's shared-memory accesses are ordered by its own arrive.  False if a bounded
// wait gave up.
template <int kOutN, int kSlots>
__device__ __forceinline__ void epilogue_acc_reader(uint32_t tmem_q, uint32_t full_bar0, uint32_t empty_addr0,
                                                    uint32_t slot_full0, uint32_t slot_empty0, uint32_t slot_buf0,
                                                    bool pair, int unit, int units, int total, int lane,
                                                    volatile int* abort_flag, int* err, int site) {
  const uint32_t row = static_cast<uint32_t>(lane) * 128u, key = static_cast<uint32_t>(lane) & 7u;
  uint32_t k = 0;  // chunks handed over so far
  int it = 0;
  for (int tile = unit; tile < total; tile += units, ++it) {
    const int acc = it & 1;
    const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
    const bool ok = mbar_wait(full_bar0 + 8u * acc, use, abort_flag, err, site);
    if (!__all_sync(0xFFFFFFFFu, ok)) return;
    tc_fence_after();
#pragma unroll 1
    for (int cc = 0; cc < kOutN; cc += 32, ++k) {
      const uint32_t slot = k % kSlots, sphase = (k / kSlots) & 1u;
      uint32_t r[32];
      tmem_ld32(tmem_q + static_cast<uint32_t>(acc * kBN + cc), r);
      const bool free_ok = mbar_wait(slot_empty0 + 8u * slot, sphase ^ 1u, abort_flag, err, site + 1);
      tmem_ld_wait();
      if (!__all_sync(0xFFFFFFFFu, free_ok)) return;
      const uint32_t dst = slot_buf0 + slot * kAccSlotBytes + row;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        st_shared_v4(dst + ((static_cast<uint32_t>(j) ^ key) << 4), r[4 * j], r[4 * j + 1], r[4 * j + 2],
                     r[4 * j + 3]);
      mbar_arrive(slot_full0 + 8u * slot);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (pair)
        mbar_arrive_cluster_relaxed(mapa_shared(empty_addr0 + 8u * acc, 0));
      else
        mbar_arrive(empty_addr0 + 8u * acc);
    }
  }
}

// Activation-backward epilogue (EPI_ACT_BWD / EPI_GLU_BWD) for the tiles of one warp (32 rows x 256
// columns of each tile, in 32-column chunks), with every global access a TMA box:
//  * SRC = ACC_TMEM: the warp reads its own TMEM lane quarter, every chunk of every tile, and hands
//    each accumulator back after its last chunk;
//  * SRC = ACC_SLOT: a helper warp for quarter 1 takes chunks c_first, c_first + c_step, ... of every
//    tile from the reader's kSlots slots (bases slot_full / slot_empty / slot_buf), never touching TMEM;
//  * the saved first-linear output of the chunk (Z, or G and U) is loaded into the warp's input
//    buffer; the next chunk's load is issued as soon as the lanes have read the current one, so it
//    overlaps the current chunk's accumulator read, arithmetic and stores;
//  * dZ (or dG, dU) and the recomputed activation H are written into the warp's output buffer and
//    stored with bulk tensor copies (clipped at the tensor edges).
// Shared-memory boxes are 32 rows x 64 bytes with 64-byte swizzle: 16-byte chunk j of row r sits at
// position j ^ ((r >> 1) & 3) of the row.
template <int EPI, int kTileM, int kOutN, int SRC, int kSlots = 2>
__device__ __forceinline__ void epilogue_act_bwd_tma(const GemmArgs& a, const EpiMaps& em, uint32_t tmem_q,
                                                     uint32_t full_bar0, uint32_t empty_addr0, uint32_t in_bar,
                                                     uint32_t buf, uint32_t slot_full, uint32_t slot_empty,
                                                     uint32_t slot_buf, int c_first, int c_step, bool pair,
                                                     int unit, int units, int total, int row_off, int lane,
                                                     volatile int* abort_flag, int* err) {
  constexpr bool kGlu = EPI == EPI_GLU_BWD;
  constexpr uint32_t kInBytes = kGlu ? 4096u : 2048u;
  const uint32_t ibuf = buf, obuf = buf + 4096u;
  const uint32_t rsw = static_cast<uint32_t>(lane) * 64u;          // this lane's row in a box
  const uint32_t rx = (static_cast<uint32_t>(lane) >> 1) & 3u;      // its 64-byte swizzle key
  const int c0 = 32 * c_first, cstep = 32 * c_step;
  struct Cursor {
    int tile, cc;
  };
  auto advance = [&](Cursor& c) {
    c.cc += cstep;
    if (c.cc >= kOutN) {
      c.cc = c0;
      c.tile += units;
    }
  };
  // A chunk is processed (and its inputs loaded) only if its rows and columns start in range.
  auto chunk = [&](const Cursor& c, int& g, int& row0, int& col) -> bool {
    if (c.tile >= total) return false;
    int mt, nt;
    decode_tile(c.tile, a, g, mt, nt);
    row0 = mt * kTileM + row_off;
    col = nt * kOutN + c.cc;
    return row0 < a.M && col < a.N;
  };
  bool pending = false;  // an input copy was issued and not yet waited for
  auto issue = [&](const Cursor& c) {
    int g, row0, col;
    if (!chunk(c, g, row0, col)) return;
    pending = true;
    if (lane == 0) {
      fence_proxy_async_smem();  // lanes' reads of the buffer precede the copy that overwrites it
      mbar_arrive_expect_tx(in_bar, kInBytes);
      tma_load_3d(ibuf, &em.m[0], in_bar, col, row0, g);
      if constexpr (kGlu) tma_load_3d(ibuf + 2048u, &em.m[1], in_bar, col, row0, g);
    }
  };
  Cursor pf{unit, c0};
  issue(pf);
  advance(pf);
  uint32_t in_phase = 0, n_stored = 0;
  const uint32_t key = static_cast<uint32_t>(lane) & 7u;
  int it = 0;
  for (int tile = unit; tile < total; tile += units, ++it) {
    const int acc = it & 1;
    if constexpr (SRC == ACC_TMEM) {
      const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
      const bool ok = mbar_wait(full_bar0 + 8u * acc, use, abort_flag, err, a.err_site + 4);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
    }
    bool aborted = false;
#pragma unroll 1
    for (int cc = c0; cc < kOutN; cc += cstep) {
      const Cursor cur{tile, cc};
      int g, row0, col;
      const bool valid = chunk(cur, g, row0, col);
      uint32_t r[32];
      if constexpr (SRC == ACC_TMEM) {
        tmem_ld32(tmem_q + static_cast<uint32_t>(acc * kBN + cc), r);
      } else {
        // every chunk passes through its slot, in range or not, so the reader's count stays in step
        const uint32_t k = static_cast<uint32_t>(it) * (kOutN / 32) + static_cast<uint32_t>(cc / 32);
        const uint32_t slot = k % kSlots;
        const bool got = mbar_wait(slot_full + 8u * slot, (k / kSlots) & 1u, abort_flag, err, a.err_site + 8);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          aborted = true;
          break;
        }
        const uint32_t src = slot_buf + slot * kAccSlotBytes + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 v = ld_shared_v4(src + ((static_cast<uint32_t>(j) ^ key) << 4));
          r[4 * j] = v.x; r[4 * j + 1] = v.y; r[4 * j + 2] = v.z; r[4 * j + 3] = v.w;
        }
        mbar_arrive(slot_empty + 8u * slot);
      }
      uint32_t zi[16], ui[16];
      if (valid) {
        const bool got = mbar_wait(in_bar, in_phase, abort_flag, err, a.err_site + 5);
        if (got) {
          in_phase ^= 1u;
          pending = false;
        }
        if (!__all_sync(0xFFFFFFFFu, got)) {
          aborted = true;
          if constexpr (SRC == ACC_TMEM) tmem_ld_wait();
          break;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t off = rsw + ((static_cast<uint32_t>(j) ^ rx) << 4);
          const uint4 zv = ld_shared_v4(ibuf + off);
          zi[4 * j] = zv.x; zi[4 * j + 1] = zv.y; zi[4 * j + 2] = zv.z; zi[4 * j + 3] = zv.w;
          if constexpr (kGlu) {
            const uint4 uv = ld_shared_v4(ibuf + 2048u + off);
            ui[4 * j] = uv.x; ui[4 * j + 1] = uv.y; ui[4 * j + 2] = uv.z; ui[4 * j + 3] = uv.w;
          }
        }
      }
      __syncwarp();
      issue(pf);
      advance(pf);
      if constexpr (SRC == ACC_TMEM) tmem_ld_wait();
      if (!valid) continue;
      uint32_t o1[16], o2[16], oh[16];
      if constexpr (kGlu) {
        if (a.act == ACT_SWIGLU)
          bwd_act_chunk<true, ACT_SWIGLU>(zi, ui, r, o1, o2, oh);
        else
          bwd_act_chunk<true, ACT_BILINEAR>(zi, ui, r, o1, o2, oh);
      } else if (a.act == ACT_GELU) {
        bwd_act_chunk<false, ACT_GELU>(zi, ui, r, o1, o2, oh);
      } else if (a.act == ACT_RELU) {
        bwd_act_chunk<false, ACT_RELU>(zi, ui, r, o1, o2, oh);
      } else {
        bwd_act_chunk<false, ACT_NONE>(zi, ui, r, o1, o2, oh);
      }
      if (lane == 0 && n_stored > 0) bulk_wait_group_read<0>();  // previous stores done reading
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t off = rsw + ((static_cast<uint32_t>(j) ^ rx) << 4);
        st_shared_v4(obuf + off, o1[4 * j], o1[4 * j + 1], o1[4 * j + 2], o1[4 * j + 3]);
        if constexpr (kGlu) st_shared_v4(obuf + 2048u + off, o2[4 * j], o2[4 * j + 1], o2[4 * j + 2], o2[4 * j + 3]);
        st_shared_v4(obuf + 4096u + off, oh[4 * j], oh[4 * j + 1], oh[4 * j + 2], oh[4 * j + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&em.m[2], obuf, col, row0, g);
        if constexpr (kGlu) tma_store_3d(&em.m[3], obuf + 2048u, col, row0, g);
        tma_store_3d(&em.m[4], obuf + 4096u, col, row0, g);
        bulk_commit_group();
      }
      ++n_stored;
    }
    if (aborted) break;
    if constexpr (SRC == ACC_TMEM) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (pair)
          mbar_arrive_cluster_relaxed(mapa_shared(empty_addr0 + 8u * acc, 0));
        else
          mbar_arrive(empty_addr0 + 8u * acc);
      }
    }
  }
  if (lane == 0) {
    bulk_wait_group_all();  // stores done before the staging memory goes away
    // after an abort an input copy may still be in flight: let it land (bounded) before the CTA
    // leaves; it completes the barrier phase with parity in_phase
    if (pending) mbar_wait_drain(in_bar, in_phase);
  }
  __syncwarp();
}

// Forward first-linear epilogue through TMA stores (EPI_ACT_BF16 / EPI_GLU_BF16), one 32-column chunk
// at a time for the warp's 32 rows: H = act(D) (or glu(gate, up)) and, when the backward's saved
// copy is requested, the pre-activation Z (or G and U), each rounded to bf16, written to the warp's
// staging boxes (64-byte swizzle) and stored with bulk tensor copies.  Maps: m[0] H, m[1] Z or G,
// m[2] U.  The staging boxes are rewritten once the previous chunk's stores have read them.
// fwd_chunk_store does one chunk from the accumulator values rz (and ru, the up columns of the gated
// form) in registers; epilogue_fwd_tma takes them from the warp's TMEM lane quarter.
template <int EPI>
__device__ __forceinline__ void fwd_chunk_store(const GemmArgs& a, const EpiMaps& em, const uint32_t (&rz)[32],
                                                const uint32_t (&ru)[32], int g, int row0, int col, uint32_t buf,
                                                uint32_t& nstore, int lane) {
  constexpr bool kGlu = EPI == EPI_GLU_BF16;
  const bool save = a.out1 != nullptr;
  const uint32_t rsw = static_cast<uint32_t>(lane) * 64u;
  const uint32_t rx = (static_cast<uint32_t>(lane) >> 1) & 3u;
  uint32_t oh[16], oz[16], ou[16];
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const float z0 = __uint_as_float(rz[e]), z1 = __uint_as_float(rz[e + 1]);
    if constexpr (kGlu) {
      const float u0 = __uint_as_float(ru[e]), u1 = __uint_as_float(ru[e + 1]);
      oh[e >> 1] = pack_bf16x2(glu_fwd(a.act, z0, u0), glu_fwd(a.act, z1, u1));
      ou[e >> 1] = pack_bf16x2(u0, u1);
    } else {
      oh[e >> 1] = pack_bf16x2(act_fwd(a.act, z0), act_fwd(a.act, z1));
    }
    oz[e >> 1] = pack_bf16x2(z0, z1);
  }
  if (lane == 0 && nstore > 0) bulk_wait_group_read<0>();
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t off = rsw + ((static_cast<uint32_t>(j) ^ rx) << 4);
    st_shared_v4(buf + off, oh[4 * j], oh[4 * j + 1], oh[4 * j + 2], oh[4 * j + 3]);
    if (save) {
      st_shared_v4(buf + 2048u + off, oz[4 * j], oz[4 * j + 1], oz[4 * j + 2], oz[4 * j + 3]);
      if constexpr (kGlu) st_shared_v4(buf + 4096u + off, ou[4 * j], ou[4 * j + 1], ou[4 * j + 2], ou[4 * j + 3]);
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_3d(&em.m[0], buf, col, row0, g);
    if (save) {
      tma_store_3d(&em.m[1], buf + 2048u, col, row0, g);
      if constexpr (kGlu) tma_store_3d(&em.m[2], buf + 4096u, col, row0, g);
    }
    bulk_commit_group();
  }
  ++nstore;
}

template <int EPI, int NC>
__device__ __forceinline__ void epilogue_fwd_tma(const GemmArgs& a, const EpiMaps& em, uint32_t tacc, int g,
                                                 int row0, int col0, uint32_t buf, uint32_t& nstore, int lane) {
  constexpr bool kGlu = EPI == EPI_GLU_BF16;
  if (row0 >= a.M) return;
#pragma unroll 1
  for (int cc = 0; cc < NC; cc += 32) {
    const int col = col0 + cc;
    if (col >= a.N) break;
    uint32_t rz[32], ru[32];
    tmem_ld32(tacc + cc, rz);
    if constexpr (kGlu) tmem_ld32(tacc + 128 + cc, ru);
    tmem_ld_wait();
    fwd_chunk_store<EPI>(a, em, rz, ru, g, row0, col, buf, nstore, lane);
  }
}

// Helper warp of the non-gated forward epilogue for TMEM lane quarter 1 (see epilogue_acc_reader): for
// every tile of the unit, chunks c_first, c_first + 2, ... of its 256 columns arrive in the reader's
// kSlots slots (bases slot_full / slot_empty / slot_buf) and leave through fwd_chunk_store, rows
// row_off + lane.
template <int EPI, int kTileM, int kOutN, int kSlots>
__device__ __forceinline__ void epilogue_fwd_helper(const GemmArgs& a, const EpiMaps& em, uint32_t buf,
                                                    uint32_t slot_full, uint32_t slot_empty, uint32_t slot_buf,
                                                    int c_first, int unit, int units, int total, int row_off,
                                                    int lane, volatile int* abort_flag, int* err) {
  const uint32_t src = slot_buf + static_cast<uint32_t>(lane) * 128u, key = static_cast<uint32_t>(lane) & 7u;
  uint32_t nstore = 0;
  int it = 0;
  for (int tile = unit; tile < total; tile += units, ++it) {
    int g, mt, nt;
    decode_tile(tile, a, g, mt, nt);
    const int row0 = mt * kTileM + row_off;
    bool aborted = false;
#pragma unroll 1
    for (int cc = 32 * c_first; cc < kOutN; cc += 64) {
      // every chunk passes through its slot, in range or not, so the reader's count stays in step
      const uint32_t k = static_cast<uint32_t>(it) * (kOutN / 32) + static_cast<uint32_t>(cc / 32);
      const uint32_t slot = k % kSlots;
      const bool got = mbar_wait(slot_full + 8u * slot, (k / kSlots) & 1u, abort_flag, err, a.err_site + 8);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        aborted = true;
        break;
      }
      uint32_t rz[32], ru[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 v = ld_shared_v4(src + slot * kAccSlotBytes + ((static_cast<uint32_t>(j) ^ key) << 4));
        rz[4 * j] = v.x; rz[4 * j + 1] = v.y; rz[4 * j + 2] = v.z; rz[4 * j + 3] = v.w;
      }
      mbar_arrive(slot_empty + 8u * slot);
      const int col = nt * kOutN + cc;
      if (row0 < a.M && col < a.N) fwd_chunk_store<EPI>(a, em, rz, ru, g, row0, col, buf, nstore, lane);
    }
    if (aborted) break;
  }
  if (lane == 0) bulk_wait_group_all();  // stores done before the staging memory goes away
  __syncwarp();
}

// Four fp32 values -> four E4M3 codes (nearest, ties to even, saturating at +-448), the first in the
// lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// FP8 first-linear epilogue (EPI_ACT_F8 / EPI_GLU_F8) of NC accumulator columns for the calling
// thread's row: H = act(alpha D) (gated: glu(alpha gate, alpha up), the up columns 128 further),
// times out_scale, rounded to E4M3 and stored with two 16-byte stores per 32 columns (N is a
// multiple of 16).
template <int EPI, int NC>
__device__ __forceinline__ void epilogue_f8_cols(const GemmArgs& a, uint32_t tacc, int g, int row, int col0) {
  const bool row_ok = row < a.M;
#pragma unroll 1
  for (int cc = 0; cc < NC; cc += 32) {
    uint32_t rz[32], ru[32];
    tmem_ld32(tacc + cc, rz);
    if constexpr (EPI == EPI_GLU_F8) tmem_ld32(tacc + 128 + cc, ru);
    tmem_ld_wait();
    const int col = col0 + cc;
    if (!row_ok || col >= a.N) continue;
    uint32_t w[8];
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      float v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float z = __uint_as_float(rz[e + k]) * a.alpha;
        float hv;
        if constexpr (EPI == EPI_GLU_F8)
          hv = glu_fwd(a.act, z, __uint_as_float(ru[e + k]) * a.alpha);
        else
          hv = act_fwd(a.act, z);
        v[k] = hv * a.out_scale;
      }
      w[e >> 2] = pack_e4m3x4(v[0], v[1], v[2], v[3]);
    }
    uint8_t* o = static_cast<uint8_t*>(a.out0) + g * a.bs0 + static_cast<int64_t>(row) * a.ld0 + col;
    *reinterpret_cast<uint4*>(o) = make_uint4(w[0], w[1], w[2], w[3]);
    if (col + 16 < a.N) *reinterpret_cast<uint4*>(o + 16) = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// fp32 epilogue through TMA stores: each 32-column chunk of the warp's 32 rows is written to one
// of the warp's two staging buffers (row `lane`, 16-byte chunk j at position j ^ (lane % 8), the
// 128-byte swizzle pattern) and stored by one lane with a bulk tensor copy; TMA clips rows and
// columns outside the output.  A buffer is rewritten only after the store issued from it two
// chunks earlier has finished reading it.
template <int NC, bool SCALE>
__device__ __forceinline__ void epilogue_f32_tma(const GemmArgs& a, const CUtensorMap* tmC, uint32_t tacc, int g,
                                                 int row0, int col0, uint32_t staging, uint32_t& nchunk,
                                                 int lane) {
  if (row0 >= a.M) return;
#pragma unroll 1
  for (int cc = 0; cc < NC; cc += 32) {
    if (col0 + cc >= a.N) break;
    const uint32_t buf = staging + (nchunk & 1u) * 4096u;
    if (lane == 0 && nchunk >= 2) bulk_wait_group_read<1>();
    __syncwarp();
    uint32_t r[32];
    tmem_ld32(tacc + cc, r);
    tmem_ld_wait();
    if constexpr (SCALE) {
#pragma unroll
      for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * a.alpha);
    }
    const uint32_t row = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_v4(row + ((static_cast<uint32_t>(j) ^ (static_cast<uint32_t>(lane) & 7u)) << 4), r[4 * j],
                   r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tmC, buf, col0 + cc, row0, g);
      bulk_commit_group();
    }
    ++nchunk;
  }
}

// One 16-column piece of this thread's TMEM lane (32x32b shape, warp-collective).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// Fused shard-sum (EPI_F32_REDUCE), one sub-tile: shard g's partial of an output tile, for the
// calling thread's row and its warp's 128 accumulator columns from `tacc`.  A unit visits the shards of an output tile consecutively and every warp
// takes the same rows and columns of each, so the row's running sum stays in the thread's
// registers: S = P_0, then S = S + P_g for g = 1, 2, ..., one fp32 add rounded to nearest per
// shard -- the order and the roundings of the stand-alone shard-sum over stored partials (E4M3
// operands: each partial is first scaled by alpha and rounded, as the partial store does).  No
// partial leaves the SM.
template <bool SCALE>
__device__ __forceinline__ void sum_partial_regs(const GemmArgs& a, uint32_t tacc, int g, float (&s)[128]) {
#pragma unroll
  for (int c = 0; c < 128; c += 16) {
    uint32_t r[16];
    tmem_ld16(tacc + static_cast<uint32_t>(c), r);
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float v = __uint_as_float(r[e]);
      if constexpr (SCALE) v = __fmul_rn(v, a.alpha);
      s[c + e] = g == 0 ? v : __fadd_rn(s[c + e], v);
    }
  }
}

// Brings the 128-byte line holding p into L2 (a hint; no fault for any address of a mapped buffer).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

// After an output tile's last shard: Y = bf16(res + S) (out1 / ld1; residual in0 / ldi, nullable)
// for the calling thread's row, 128 columns from col0, straight from the registers.  Rows past
// M and columns past N are not written (N % 8 = 0: eight columns are all in or all out).  Y may be
// the residual itself (a layer stack updates Z in place), so each residual load must precede the
// stores that could overwrite it: the residual is read 16 columns at a time, two independent
// loads in flight, before those columns are stored (four would need registers that the 128 sums
// leave no room for).
__device__ __forceinline__ void store_sum_row(const GemmArgs& a, int row, int col0, const float (&s)[128]) {
  if (row >= a.M) return;
  uint16_t* y = static_cast<uint16_t*>(a.out1) + static_cast<int64_t>(row) * a.ld1 + col0;
  const uint16_t* res = static_cast<const uint16_t*>(a.in0);
  const uint16_t* rp = res ? res + static_cast<int64_t>(row) * a.ldi + col0 : nullptr;
  constexpr int kResGroup = 2;
#pragma unroll
  for (int c0 = 0; c0 < 128; c0 += 8 * kResGroup) {
    uint4 w[kResGroup];
#pragma unroll
    for (int q = 0; q < kResGroup; ++q) {
      const int c = c0 + 8 * q;
      w[q] = (rp && col0 + c < a.N) ? __ldcg(reinterpret_cast<const uint4*>(rp + c))
                                                : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < kResGroup; ++q) {
      const int c = c0 + 8 * q;
      if (col0 + c >= a.N) continue;
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = s[c + e];
      if (rp) {
        // residual first, then the sum, as in the stand-alone shard-sum: res + S, one rounding
        v[0] = bf16lo(w[q].x) + v[0]; v[1] = bf16hi(w[q].x) + v[1];
        v[2] = bf16lo(w[q].y) + v[2]; v[3] = bf16hi(w[q].y) + v[3];
        v[4] = bf16lo(w[q].z) + v[4]; v[5] = bf16hi(w[q].z) + v[5];
        v[6] = bf16lo(w[q].w) + v[6]; v[7] = bf16hi(w[q].w) + v[7];
      }
      store8_bf16(y + c, v);
    }
  }
}

// Split tiles of the fused shard-sum (fused_tile).  A partial slot holds one shard's 256 x 256 fp32
// partial of one output tile (256 KiB) in thread order: 16-byte piece q (columns 4q .. 4q+3 of the
// thread's 128) of lane l of epilogue warp w of CTA r at ((r * 8 + w) * 32 + q) * 32 + l.  A warp's
// piece q is then 512 contiguous bytes, and each warp's block (16 KiB) is contiguous.  The slot's
// counter reaches kSlotWriters (every epilogue warp of both CTAs) once all pieces are written.
constexpr int64_t kSlotBytes = 256 * 256 * 4;
constexpr uint32_t kSlotWriters = 16;
constexpr uint32_t kSlotWarpBytes = 32 * 32 * 16;

// Split tile: this thread's 128 accumulator columns of one shard into its pieces of the shard's slot
// (w: its piece 0), scaled and rounded as the partial store does.
template <bool SCALE>
__device__ __forceinline__ void store_partial_slot(const GemmArgs& a, uint32_t tacc, uint4* w) {
#pragma unroll
  for (int c = 0; c < 128; c += 16) {
    uint32_t r[16];
    tmem_ld16(tacc + static_cast<uint32_t>(c), r);
    tmem_ld_wait();
    if constexpr (SCALE) {
#pragma unroll
      for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__fmul_rn(__uint_as_float(r[e]), a.alpha));
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      __stcg(w + (c / 4 + q) * 32, make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]));
  }
}

// Helper, once the warp's pieces of a slot are written: counts the warp in, with release semantics at
// GPU scope (the lanes' stores precede lane 0's fence through the warp barrier).
__device__ __forceinline__ void publish_slot(uint32_t* counter, int lane) {
  __syncwarp();
  if (lane == 0) {
    __threadfence();
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
  }
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Head: bounded wait until every helper warp has written its pieces of a slot (lane 0 polls; then
// every lane takes its own acquire of the counter).
__device__ __forceinline__ bool wait_slot(const uint32_t* counter, volatile int* abort_flag, int* err, int site,
                                          int lane) {
  bool ok = true;
  if (lane == 0) {
    uint64_t t0 = 0;
    for (uint32_t it = 0; ld_acquire_u32(counter) < kSlotWriters; ++it) {
      if ((it & 63u) == 63u) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        const uint64_t now = global_timer_ns();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > kWaitTimeoutNs) {
          *abort_flag = 1;
          atomicCAS(err, 0, site);
          ok = false;
          break;
        }
      }
    }
  }
  ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
  if (ok) (void)ld_acquire_u32(counter);
  return ok;
}

// Untiled bulk copy global -> this CTA's shared memory, completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Head: adds one shard's partial from its slot into the thread's sums, in shard order (g = 0: the
// sums start from it).  The warp's
// 16 KiB block is brought into `buf` (shared memory the warp owns) by one bulk copy on the warp's
// barrier `bar` (phase `ph`), then each lane adds its 32 pieces.  False if the wait gave up.
template <bool FIRST>
__device__ __forceinline__ bool add_partial_slot(const uint8_t* block, uint32_t buf, uint32_t bar, uint32_t ph,
                                                 int lane, volatile int* abort_flag, int* err, int site,
                                                 float (&s)[128]) {
  __syncwarp();  // the lanes' reads of the previous block are done
  if (lane == 0) {
    fence_proxy_async_smem();    // ... before the copy that overwrites them
    fence_proxy_async_global();  // the helpers' writes, acquired above, precede the copy's reads
    mbar_arrive_expect_tx(bar, kSlotWarpBytes);
    bulk_load(buf, block, kSlotWarpBytes, bar);
  }
  const bool ok = mbar_wait(bar, ph, abort_flag, err, site);
  if (!__all_sync(0xFFFFFFFFu, ok)) return false;
#pragma unroll
  for (int q = 0; q < 32; ++q) {
    const uint4 v = ld_shared_v4(buf + static_cast<uint32_t>((q * 32 + lane) * 16));
    if constexpr (FIRST) {
      s[4 * q] = __uint_as_float(v.x);
      s[4 * q + 1] = __uint_as_float(v.y);
      s[4 * q + 2] = __uint_as_float(v.z);
      s[4 * q + 3] = __uint_as_float(v.w);
    } else {
      s[4 * q] = __fadd_rn(s[4 * q], __uint_as_float(v.x));
      s[4 * q + 1] = __fadd_rn(s[4 * q + 1], __uint_as_float(v.y));
      s[4 * q + 2] = __fadd_rn(s[4 * q + 2], __uint_as_float(v.z));
      s[4 * q + 3] = __fadd_rn(s[4 * q + 3], __uint_as_float(v.w));
    }
  }
  return true;
}

// Head of a split tile: sums the tile's slots (block: this warp's block in slot 0, the next slots
// kSlotBytes apart; counters cnt[g]) in shard order through `buf`, the warp's 16 KiB of shared
// memory, then writes Y for the thread's row.  A function of its own, so that its 128 sums are
// allocated apart from the whole-tile loop's.  False if a wait gave up.
static __device__ __noinline__ bool head_sum_slots(const GemmArgs& a, const uint8_t* block, const uint32_t* cnt, uint32_t buf,
                                            uint32_t bar, int row, int col0, int lane, volatile int* abort_flag,
                                            int* err) {
  float s[128];
  bool ok = wait_slot(cnt, abort_flag, err, a.err_site + 6, lane) &&
            add_partial_slot<true>(block, buf, bar, 0u, lane, abort_flag, err, a.err_site + 7, s);
  for (int g = 1; ok && g < a.batches; ++g)
    ok = wait_slot(cnt + g, abort_flag, err, a.err_site + 6, lane) &&
         add_partial_slot<false>(block + static_cast<int64_t>(g) * kSlotBytes, buf, bar, static_cast<uint32_t>(g) & 1u,
                                 lane, abort_flag, err, a.err_site + 7, s);
  if (ok) store_sum_row(a, row, col0, s);
  return ok;
}

// F8: operands are E4M3 codes (kind::f8f6f4), 128 elements per 128-byte K step.
template <int EPI, bool A_MN, bool B_MN, bool PAIR, bool F8 = false>
__global__ void __launch_bounds__(bound_threads<EPI>(), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ EpiMaps em, const GemmArgs args) {
  using R = Ring<PAIR, EPI>;
  constexpr int S = R::kStages;
  static_assert(!F8 || (!A_MN && !B_MN && PAIR), "FP8 operands: K-major, CTA pair");
  static_assert(is_act_f8(EPI) ? F8 : (!F8 || EPI == EPI_F32_STORE || EPI == EPI_F32_REDUCE),
                "the E4M3 epilogues go with FP8 operands, which take only those and the fp32 ones");
  constexpr bool kGatedB = is_gated_b(EPI);
  constexpr int kOutN = kGatedB ? 128 : kBN;
  constexpr int kKe = F8 ? 128 : kBK;  // K elements per stage (always 128 bytes per row)
  constexpr uint32_t kIdesc =
      F8 ? idesc_e4m3_f32(R::kTileM, kBN, A_MN, B_MN) : idesc_bf16_f32(R::kTileM, kBN, A_MN, B_MN);
  // barrier indices in the control block
  constexpr int kBarFull = 0, kBarEmpty = S, kBarTmemFull = 2 * S, kBarTmemEmpty = 2 * S + 2,
                kBarDrain = 2 * S + 4, kBarEpiIn = 2 * S + 5;  // kBarEpiIn: one per epilogue warp
  // the peer CTA's producer reports how many ring uses it issued (CTA pair, leader's barrier)
  constexpr int kBarPeerCount = kBarEpiIn + epi_warps<EPI>();
  // helper warps: their input barriers and the accumulator slots of lane quarter 1 (full, empty)
  constexpr int kSlots = kAccSlots;
  constexpr int kBarHelperIn = kBarPeerCount + 1, kBarSlotFull = kBarHelperIn + 2,
                kBarSlotEmpty = kBarSlotFull + kSlots;
  static_assert(8 * (kBarSlotEmpty + kSlots) <= 512, "barriers overlap the TMEM slot");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 516);
  volatile uint32_t* peer_issued = reinterpret_cast<volatile uint32_t*>(smem + 520);  // written by the peer
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t stage0 = smem_u32(smem + kCtrlBytes);
  auto bar = [bar0](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;  // 0 = leader of the pair
  const bool leader = rank == 0;
  const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int units = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  int* err = &g_gemm_err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarTmemFull + i), 1);
      mbar_init(bar(kBarTmemEmpty + i), (PAIR ? 2 : 1) * epi_warps<EPI>());
    }
    mbar_init(bar(kBarDrain), 1);
    for (int e = 0; e < epi_warps<EPI>(); ++e) mbar_init(bar(kBarEpiIn + e), 1);
    mbar_init(bar(kBarPeerCount), 1);
    if constexpr (helper_warps<EPI>() > 0) {
      for (int i = 0; i < 2; ++i) mbar_init(bar(kBarHelperIn + i), 1);
      for (int i = 0; i < kSlots; ++i) {
        mbar_init(bar(kBarSlotFull + i), 32);   // every lane of the reader arrives
        mbar_init(bar(kBarSlotEmpty + i), 32);  // every lane of the helper arrives
      }
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
    if constexpr (EPI == EPI_F32_STORE) tma_prefetch_map(&em.m[0]);
    if constexpr (is_act_fwd(EPI)) {
      tma_prefetch_map(&em.m[0]);
      if (args.out1) tma_prefetch_map(&em.m[1]);
      if (EPI == EPI_GLU_BF16 && args.out1) tma_prefetch_map(&em.m[2]);
    }
    if constexpr (is_act_bwd(EPI))
      for (int i = 0; i < 5; ++i)
        if ((i != 1 && i != 3) || EPI == EPI_GLU_BWD) tma_prefetch_map(&em.m[i]);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();  // barrier initialisation visible to the peer before any remote signal
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = args.batches * args.m_tiles * args.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs of a pair load their own halves)
      uint32_t s = 0, ph = 0, armed = 0, armed_ph = 0, issued = 0;
      bool ok = true;
      int g, mt, nt;
      for (int sq = 0; ok && tile_at<EPI>(sq, args, unit, units, g, mt, nt); ++sq) {
        const int m0 = mt * R::kTileM + static_cast<int>(rank) * kBM + args.a_row_off;
        const int n0 = nt * kOutN + args.b_row_off + ((PAIR && !kGatedB) ? static_cast<int>(rank) * 128 : 0);
        const int ga = g * args.a_bmul, gb = g * args.b_bmul;
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait(bar(kBarEmpty + s), ph ^ 1u, abort_flag, err, args.err_site + 1)) {
            ok = false;
            break;
          }
          const uint32_t sa = stage0 + s * R::kStageBytes, sb = sa + R::kABytes;
          const uint32_t fb_local = bar(kBarFull + s);
          const int k0 = kb * kKe;
          if constexpr (PAIR) {
            // the leader's full barrier counts the bytes of both CTAs
            const uint32_t fb = mapa_shared(fb_local, 0);
            if (leader) mbar_arrive_expect_tx(fb_local, 2u * R::kStageBytes);
            if constexpr (!A_MN) {
              tma_load_3d_pair(sa, &tmA, fb, k0, m0, ga);
            } else {
              tma_load_3d_pair(sa, &tmA, fb, m0, k0, ga);
              tma_load_3d_pair(sa + 8192, &tmA, fb, m0 + 64, k0, ga);
            }
            if constexpr (kGatedB) {
              tma_load_4d_pair(sb, &tmB, fb, k0, n0, static_cast<int>(rank), g);
            } else if constexpr (!B_MN) {
              tma_load_3d_pair(sb, &tmB, fb, k0, n0, gb);
            } else {
              tma_load_3d_pair(sb, &tmB, fb, n0, k0, gb);
              tma_load_3d_pair(sb + 8192, &tmB, fb, n0 + 64, k0, gb);
            }
          } else {
            mbar_arrive_expect_tx(fb_local, R::kStageBytes);
            armed |= 1u << s;
            armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
            if constexpr (!A_MN) {
              tma_load_3d(sa, &tmA, fb_local, k0, m0, ga);
            } else {
              tma_load_3d(sa, &tmA, fb_local, m0, k0, ga);
              tma_load_3d(sa + 8192, &tmA, fb_local, m0 + 64, k0, ga);
            }
            if constexpr (kGatedB) {
              tma_load_4d(sb, &tmB, fb_local, k0, n0, 0, g);
              tma_load_4d(sb + 16384, &tmB, fb_local, k0, n0, 1, g);
            } else if constexpr (!B_MN) {
              tma_load_3d(sb, &tmB, fb_local, k0, n0, gb);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j) tma_load_3d(sb + 8192 * j, &tmB, fb_local, n0 + 64 * j, k0, gb);
            }
          }
          ++issued;
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if constexpr (PAIR) {
        // Both CTAs' copies complete on the leader's barriers: the peer tells the leader how many ring
        // uses it issued, and the leader, if anything was left unconsumed (an abort on either side),
        // waits until every copy of both CTAs has landed before the pair leaves at the final
        // cluster barrier.
        if (!leader) {
          st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t*>(peer_issued)), 0), issued);
          mbar_arrive_cluster(mapa_shared(bar(kBarPeerCount), 0));
        } else if (mbar_wait_cluster_acquire(bar(kBarPeerCount), 0, kPeerCountTimeoutNs)) {
          const uint32_t peer = *peer_issued;
          if (!ok || peer != issued || *abort_flag) drain_pair_ring<S>(bar(kBarFull), issued, peer, R::kStageBytes);
        } else {
          // the peer never reported (its GPU side stopped making progress): give its copies time
          const uint64_t t0 = global_timer_ns();
          while (global_timer_ns() - t0 < kPeerCopyGraceNs) {
          }
        }
      } else if (!ok) {
        // let this CTA's copies still in flight land before the CTA leaves
        for (int i = 0; i < S; ++i)
          if ((armed >> i) & 1u) mbar_wait_drain(bar(kBarFull + i), (armed_ph >> i) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (the leader CTA of a pair issues for both)
      uint32_t s = 0, ph = 0;
      bool ok = true;
      const int nsub = unit_subtiles<EPI>(args, unit, units);
      for (int it = 0; ok && it < nsub; ++it) {
        const uint32_t idesc = kIdesc;
        const int acc = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
        if (!mbar_wait(bar(kBarTmemEmpty + acc), use ^ 1u, abort_flag, err, args.err_site + 2)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait(bar(kBarFull + s), ph, abort_flag, err, args.err_site + 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = stage0 + s * R::kStageBytes, sb = sa + R::kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = A_MN ? sdesc_sw128(sa + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(sb + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(sb + kk * 32, 16, 1024);
            if constexpr (F8)
              umma_f8_pair(d_tmem, ad, bd, idesc, static_cast<uint32_t>((kb | kk) != 0));
            else if constexpr (PAIR)
              umma_bf16_pair(d_tmem, ad, bd, idesc, static_cast<uint32_t>((kb | kk) != 0));
            else
              umma_bf16(d_tmem, ad, bd, idesc, static_cast<uint32_t>((kb | kk) != 0));
          }
          if constexpr (PAIR)
            umma_commit_pair_multicast(bar(kBarEmpty + s), 0x3);
          else
            umma_commit(bar(kBarEmpty + s));
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          umma_commit_pair_multicast(bar(kBarTmemFull + acc), 0x3);
        else
          umma_commit(bar(kBarTmemFull + acc));
      }
      // all MMAs this thread issued have completed once the drain barrier flips
      if constexpr (PAIR)
        umma_commit_pair(bar(kBarDrain));
      else
        umma_commit(bar(kBarDrain));
      mbar_wait_drain(bar(kBarDrain), 0);
    }
  } else {
    // ---------------- epilogue warps: TMEM lane quarter = warp % 4; with two warps per quarter (the
    // fused shard-sum) warps 2-5 take the first and warps 6-9 the second half of the columns
    constexpr int kParts = epi_warps<EPI>() / 4;
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    constexpr int kHalfOut = kOutN / kParts;
    const int row_in_tile = static_cast<int>(rank) * kBM + quarter * 32 + lane;
    const uint32_t staging = stage0 + S * R::kStageBytes + static_cast<uint32_t>(warp - 2) * 8192u;
    uint32_t nchunk = 0;
    if constexpr (is_act_bwd(EPI)) {
      // warps 2-4: lane quarters 2, 3, 0 in full; warp 5 (quarter 1, beside the MMA issuer) only moves
      // its accumulator into two slots; helper warps 6 and 7 take the quarter's even and odd chunks
      const uint32_t ebase = stage0 + S * R::kStageBytes;
      const uint32_t slots = ebase + 5u * kActBwdWarpBytes;
      const int q1_row = static_cast<int>(rank) * kBM + 32;
      if (warp == 5) {
        epilogue_acc_reader<kOutN, kSlots>(tmem_base + (1u << (5 + 16)), bar(kBarTmemFull), bar(kBarTmemEmpty),
                                           bar(kBarSlotFull), bar(kBarSlotEmpty), slots, PAIR, unit, units, total,
                                           lane, abort_flag, err, args.err_site + 9);
      } else if (warp < 5) {
        epilogue_act_bwd_tma<EPI, R::kTileM, kOutN, ACC_TMEM>(
            args, em, tmem_base + (static_cast<uint32_t>(quarter * 32) << 16), bar(kBarTmemFull), bar(kBarTmemEmpty),
            bar(kBarEpiIn + (warp - 2)), ebase + static_cast<uint32_t>(warp - 2) * kActBwdWarpBytes, 0u, 0u, 0u, 0, 1,
            PAIR, unit, units, total, static_cast<int>(rank) * kBM + quarter * 32, lane, abort_flag, err);
      } else {
        const int h = warp - 6;
        epilogue_act_bwd_tma<EPI, R::kTileM, kOutN, ACC_SLOT, kSlots>(
            args, em, 0u, 0u, 0u, bar(kBarHelperIn + h), ebase + static_cast<uint32_t>(3 + h) * kActBwdWarpBytes,
            bar(kBarSlotFull), bar(kBarSlotEmpty), slots, h, 2, PAIR, unit, units, total, q1_row, lane, abort_flag,
            err);
      }
    } else if (EPI == EPI_ACT_BF16 && warp >= 5) {
      // non-gated forward activation: warp 5 moves lane quarter 1's accumulator into the slots and
      // helper warps 6 and 7 do its even and odd chunks
      if constexpr (EPI == EPI_ACT_BF16) {
      const uint32_t ebase = stage0 + S * R::kStageBytes;
      const uint32_t slots = ebase + 5u * kFwdActWarpBytes;
      if (warp == 5) {
        epilogue_acc_reader<kOutN, kSlots>(tmem_base + (1u << (5 + 16)), bar(kBarTmemFull), bar(kBarTmemEmpty),
                                           bar(kBarSlotFull), bar(kBarSlotEmpty), slots, PAIR, unit, units, total,
                                           lane, abort_flag, err, args.err_site + 9);
      } else {
        const int h = warp - 6;
        epilogue_fwd_helper<EPI, R::kTileM, kOutN, kSlots>(
            args, em, ebase + static_cast<uint32_t>(3 + h) * kFwdActWarpBytes, bar(kBarSlotFull), bar(kBarSlotEmpty),
            slots, h, unit, units, total, static_cast<int>(rank) * kBM + 32, lane, abort_flag, err);
      }
      }
    } else if constexpr (EPI == EPI_F32_REDUCE) {
      // fused shard-sum (fused_tile): per output tile of the unit, its shards in order; the running
      // sums of the thread's row (its warp's 128 columns) in registers; the unit's k-th sub-tile is in
      // accumulator k % 2.
      float s[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) s[i] = 0.0f;  // every shard 0 overwrites it
      uint32_t k = 0;
      bool ok = true;
      const int ew = warp - 2;
      const uint32_t tq = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(half * kHalfOut);
      // whole tiles (fused_tile: role FT_WHOLE), all shards in registers, then Y; the accumulators are
      // handed back as they are read, so the sum goes out while the next tile's shards run
      const int tiles = args.m_tiles * args.n_tiles, full = tiles / units, rest = tiles - full * units;
      const int nwhole = full + ((args.split <= 1 && unit < rest) ? 1 : 0);
      for (int o = 0; ok && o < nwhole; ++o) {
        int gb, mt, nt;
        decode_tile(o * units + unit, args, gb, mt, nt);
        for (int g = 0; ok && g < args.batches; ++g, ++k) {
          if (g == args.batches - 1 && args.in0) {
            // the residual row segment this thread adds at the end, into L2 while the last shard runs
            const int row = mt * R::kTileM + row_in_tile, col0 = nt * kOutN + half * kHalfOut;
            if (row < args.M) {
              const uint16_t* rp = static_cast<const uint16_t*>(args.in0) + static_cast<int64_t>(row) * args.ldi + col0;
              for (int c = 0; c < kHalfOut && col0 + c < args.N; c += 64) prefetch_l2(rp + c);
            }
          }
          const uint32_t acc = k & 1u;
          ok = mbar_wait(bar(kBarTmemFull + acc), (k >> 1) & 1u, abort_flag, err, args.err_site + 4);
          if (!__all_sync(0xFFFFFFFFu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          sum_partial_regs<F8>(args, tq + acc * kBN, g, s);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (PAIR)
              mbar_arrive_cluster_relaxed(mapa_shared(bar(kBarTmemEmpty + acc), 0));
            else
              mbar_arrive(bar(kBarTmemEmpty + acc));
          }
        }
        if (ok) store_sum_row(args, mt * R::kTileM + row_in_tile, nt * kOutN + half * kHalfOut, s);
      }
      // the unit's share of a split tile of the last round: every unit of the tile, its head included,
      // writes its shards' partials to their slots straight from TMEM; the head then sums all the
      // tile's slots in shard order through this warp's part of its operand ring, idle by then (all
      // of the unit's products have completed), and writes Y
      FusedTile f;
      if (ok && args.split > 1 && fused_tile(full, args, unit, units, f)) {
        const int64_t wofs = static_cast<int64_t>(rank * 8 + ew) * kSlotWarpBytes;  // this warp's block in a slot
        for (int g = f.lo; ok && g < f.hi; ++g, ++k) {
          const uint32_t acc = k & 1u;
          ok = mbar_wait(bar(kBarTmemFull + acc), (k >> 1) & 1u, abort_flag, err, args.err_site + 4);
          if (!__all_sync(0xFFFFFFFFu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          store_partial_slot<F8>(args, tq + acc * kBN,
                                 reinterpret_cast<uint4*>(static_cast<uint8_t*>(args.part) +
                                                          static_cast<int64_t>(f.slot0 + g) * kSlotBytes + wofs) +
                                     lane);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (PAIR)
              mbar_arrive_cluster_relaxed(mapa_shared(bar(kBarTmemEmpty + acc), 0));
            else
              mbar_arrive(bar(kBarTmemEmpty + acc));
          }
          publish_slot(args.flags + f.slot0 + g, lane);
        }
        if (ok && f.role == FT_HEAD) {
          const int row = f.mt * R::kTileM + row_in_tile, col0 = f.nt * kOutN + half * kHalfOut;
          if (args.in0 && row < args.M) {
            const uint16_t* rp = static_cast<const uint16_t*>(args.in0) + static_cast<int64_t>(row) * args.ldi + col0;
            for (int c = 0; c < kHalfOut && col0 + c < args.N; c += 64) prefetch_l2(rp + c);
          }
          ok = head_sum_slots(args, static_cast<const uint8_t*>(args.part) + static_cast<int64_t>(f.slot0) * kSlotBytes + wofs,
                              args.flags + f.slot0, stage0 + static_cast<uint32_t>(ew) * kSlotWarpBytes,
                              bar(kBarEpiIn + ew), row, col0, lane, abort_flag, err);
        }
      }
    } else {
      int g, mt, nt;
      for (int it = 0; tile_at<EPI>(it, args, unit, units, g, mt, nt); ++it) {
        const int acc = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
        const bool ok = mbar_wait(bar(kBarTmemFull + acc), use, abort_flag, err, args.err_site + 4);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
        tc_fence_after();
        const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                              static_cast<uint32_t>(acc * kBN + half * kHalfOut);
        if constexpr (EPI == EPI_F32_STORE)
          epilogue_f32_tma<kHalfOut, F8>(args, &em.m[0], tacc, g, mt * R::kTileM + row_in_tile - lane,
                                         nt * kOutN + half * kHalfOut, staging, nchunk, lane);
        else if constexpr (is_act_f8(EPI))
          epilogue_f8_cols<EPI, kHalfOut>(args, tacc, g, mt * R::kTileM + row_in_tile, nt * kOutN + half * kHalfOut);
        else if constexpr (is_act_fwd(EPI))
          epilogue_fwd_tma<EPI, kHalfOut>(
              args, em, tacc, g, mt * R::kTileM + row_in_tile - lane, nt * kOutN + half * kHalfOut,
              stage0 + S * R::kStageBytes +
                  static_cast<uint32_t>(warp - 2) * (EPI == EPI_ACT_BF16 ? kFwdActWarpBytes : kFwdWarpBytes),
              nchunk, lane);
        else
          epilogue_cols<EPI, kHalfOut>(args, tacc, g, mt * R::kTileM + row_in_tile, nt * kOutN + half * kHalfOut);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster_relaxed(mapa_shared(bar(kBarTmemEmpty + acc), 0));
          else
            mbar_arrive(bar(kBarTmemEmpty + acc));
        }
      }
    }
    if constexpr (EPI == EPI_F32_STORE || is_act_fwd(EPI)) {
      if (lane == 0) bulk_wait_group_all();  // stores done before the staging memory goes away
      __syncwarp();
    }
  }

  tc_fence_before();
  if constexpr (PAIR)
    cluster_sync();  // no CTA of the pair leaves while the other may still touch its memory
  else
    __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Launches one GEMM: one CTA (or CTA pair) per SM (pair), persistent over the tiles.
template <int EPI, bool A_MN, bool B_MN, bool F8 = false>
cudaError_t launch_gemm_t(const CUtensorMap& ta, const CUtensorMap& tb, const EpiMaps& em,
                          const GemmArgs& args, cudaStream_t st) {
  constexpr bool P = kPairMma;
  auto fn = gemm_kernel<EPI, A_MN, B_MN, P, F8>;
  constexpr int smem = smem_bytes<P, EPI>();
  static_assert(smem <= 232448, "shared memory beyond the per-CTA limit");
  // Co-resident CTAs (single) or clusters (pair), per device: the shared-memory opt-in is an
  // attribute of the function on one device and the occupancy is queried there.  0 = not set up.
  static std::atomic<int> max_units_of[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int max_units = max_units_of[dev].load(std::memory_order_acquire);
  if (max_units == 0) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if constexpr (P) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(block_threads<EPI>());
      cfg.dynamicSmemBytes = smem;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
      if (e != cudaSuccess) return e;
      if (n < 1) return cudaErrorInvalidConfiguration;
      max_units = n;
    } else {
      int sms = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      max_units = sms;
    }
    max_units_of[dev].store(max_units, std::memory_order_release);
  }
  // The fused shard-sum's units own output tiles with all their shards; a launch with fewer tiles
  // than units gives each tile up to t units (one per group of shards, fused_tile), and so does a
  // last round of at most half as many tiles as units, when `part` can hold their partial slots.
  GemmArgs a = args;
  const int64_t tiles = int64_t(EPI == EPI_F32_REDUCE ? 1 : args.batches) * args.m_tiles * args.n_tiles;
  if (tiles == 0 || args.batches == 0) return cudaSuccess;
  int units = static_cast<int>(tiles < max_units ? tiles : max_units);
  a.split = 1;
  a.flags = nullptr;
  if constexpr (EPI == EPI_F32_REDUCE) {
    const int64_t t = args.batches;
    if (t > 1 && tiles < max_units) units = static_cast<int>(tiles * t < max_units ? tiles * t : max_units);
    const int64_t rest = tiles % units;
    const int64_t split = rest > 0 ? (t < units / rest ? t : units / rest) : 1;
    const int64_t slots = rest * t;
    if (split >= 2 && a.part && a.part_bytes >= slots * (kSlotBytes + 4)) {
      a.split = static_cast<int32_t>(split);
      a.flags = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.part) + slots * kSlotBytes);
      e = cudaMemsetAsync(a.flags, 0, static_cast<size_t>(slots) * 4, st);
      if (e != cudaSuccess) return e;
    } else if (tiles < units) {
      units = static_cast<int>(tiles);
    }
  }
  if constexpr (P) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * units);
    cfg.blockDim = dim3(block_threads<EPI>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, ta, tb, em, a);
  } else {
    fn<<<units, block_threads<EPI>(), smem, st>>>(ta, tb, em, a);
    return cudaGetLastError();
  }
}

static inline cudaError_t take_error_word(int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemm_err, sizeof(int));
  if (e != cudaSuccess) return e;
  *code = v;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_gemm_err, &zero, sizeof(int));
  }
  return e;
}

}  // namespace dm
