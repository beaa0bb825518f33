// gemm.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a with fused epilogues.
//
// One CTA per SM loops over output tiles.  Warp roles:
//   warp 0 (one lane)  TMA producer: loads the A tile (128 x 64) and B tile (256 x 64) of each
//                      K step into a 4-stage shared-memory ring (128-byte swizzle).
//   warp 1 (one lane)  MMA issuer: tcgen05.mma 128x256x16 into one of two TMEM accumulators
//                      (2 x 256 fp32 columns), commits to the ring's "empty" barriers and to
//                      the accumulator's "full" barrier.  Warp 1 also owns TMEM alloc/dealloc.
//   warps 2-5          epilogue: tcgen05.ld of the accumulator (each warp reads its 32-lane
//                      quarter, one row per thread), applies the epilogue and writes global
//                      memory, then releases the accumulator so tile i+1's epilogue overlaps
//                      tile i+2's main loop.
// Every wait is bounded (ptx.cuh); on expiry the CTA drains what it has in flight, frees TMEM
// and returns, leaving a code in the translation unit's error word.
#pragma once
#include <cuda_bf16.h>

#include "actfn.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dm {

// Device error word of the GEMM kernels of the including translation unit.
static __device__ int g_gemm_err;

constexpr int kABytes = kBM * kBK * 2;        // 16 KB
constexpr int kBBytes = kBN * kBK * 2;        // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kCtrlBytes = 1024;
constexpr int kSmemBytes = 1024 /* alignment slack */ + kCtrlBytes + kStages * kStageBytes;
constexpr int kTmemCols = 2 * kBN;
constexpr int kGroupM = 8;  // tiles are visited in groups of 8 M-tiles for L2 reuse of B tiles
constexpr uint64_t kDrainTimeoutNs = 200000000ull;

// Barrier indices in the control block.
constexpr int kBarFull = 0;                 // [kStages]
constexpr int kBarEmpty = kStages;          // [kStages]
constexpr int kBarTmemFull = 2 * kStages;   // [2]
constexpr int kBarTmemEmpty = 2 * kStages + 2;  // [2]
constexpr int kBarDrain = 2 * kStages + 4;

__device__ __forceinline__ void decode_tile(int tile, const GemmArgs& a, int& g, int& mt, int& nt) {
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

// Bounded wait that ignores the abort flag (used while draining after an abort).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kDrainTimeoutNs) return;
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

// Epilogue of one 128 x kOutN tile for the calling thread's row.  `tacc` addresses this warp's
// TMEM lane quarter at column 0 of the accumulator.  Every lane executes the TMEM loads;
// only stores are masked.
template <int EPI>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& a, uint32_t tacc, int g, int row,
                                              int col0) {
  const bool row_ok = row < a.M;
  if constexpr (EPI == EPI_GLU_BF16) {
#pragma unroll 1
    for (int cc = 0; cc < 128; cc += 32) {
      uint32_t rg[32], ru[32];
      tmem_ld32(tacc + cc, rg);
      tmem_ld32(tacc + 128 + cc, ru);
      tmem_ld_wait();
      const int col = col0 + cc;
      if (!row_ok) continue;
      uint16_t* o0 = static_cast<uint16_t*>(a.out0) + g * a.bs0 + static_cast<int64_t>(row) * a.ld0 + col;
      uint16_t* o1 = a.out1 ? static_cast<uint16_t*>(a.out1) + g * a.bs1 + static_cast<int64_t>(row) * a.ld1 + col
                            : nullptr;
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
    for (int cc = 0; cc < kBN; cc += 32) {
      uint32_t r[32];
      tmem_ld32(tacc + cc, r);
      tmem_ld_wait();
      const int col = col0 + cc;
      if (!row_ok || col >= a.N) continue;
      const int64_t rowoff = static_cast<int64_t>(row);
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
      } else if constexpr (EPI == EPI_F32_STORE || EPI == EPI_F32_ACCUM) {
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
      } else if constexpr (EPI == EPI_ACT_BWD) {
        const uint16_t* zi = static_cast<const uint16_t*>(a.in0) + g * a.bsi + rowoff * a.ldi + col;
        uint16_t* o0 = static_cast<uint16_t*>(a.out0) + g * a.bs0 + rowoff * a.ld0 + col;
        uint16_t* o1 = static_cast<uint16_t*>(a.out1) + g * a.bs1 + rowoff * a.ld1 + col;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          if (col + 8 * s >= a.N) break;
          float z[8], dz[8], hv[8];
          load8_bf16(zi + 8 * s, z);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            dz[e] = __uint_as_float(r[8 * s + e]) * act_grad(a.act, z[e]);
            hv[e] = act_fwd(a.act, z[e]);
          }
          store8_bf16(o0 + 8 * s, dz);
          store8_bf16(o1 + 8 * s, hv);
        }
      } else if constexpr (EPI == EPI_GLU_BWD) {
        const uint16_t* gi = static_cast<const uint16_t*>(a.in0) + g * a.bsi + rowoff * a.ldi + col;
        uint16_t* o0 = static_cast<uint16_t*>(a.out0) + g * a.bs0 + rowoff * a.ld0 + col;
        uint16_t* o1 = static_cast<uint16_t*>(a.out1) + g * a.bs1 + rowoff * a.ld1 + col;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          if (col + 8 * s >= a.N) break;
          float gv[8], uv[8], dg[8], du[8], hv[8];
          load8_bf16(gi + 8 * s, gv);
          load8_bf16(gi + a.offi + 8 * s, uv);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            glu_bwd(a.act, gv[e], uv[e], __uint_as_float(r[8 * s + e]), dg[e], du[e], hv[e]);
          store8_bf16(o0 + 8 * s, dg);
          store8_bf16(o0 + a.off0 + 8 * s, du);
          store8_bf16(o1 + 8 * s, hv);
        }
      }
    }
  }
}

template <int EPI, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmArgs args) {
  constexpr bool kGatedB = (EPI == EPI_GLU_BF16);
  constexpr int kOutN = kGatedB ? 128 : kBN;
  constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, kBN, A_MN, B_MN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 516);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t stage0 = smem_u32(smem + kCtrlBytes);
  auto bar = [bar0](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* err = &g_gemm_err;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarTmemFull + i), 1);
      mbar_init(bar(kBarTmemEmpty + i), 4);
    }
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = args.batches * args.m_tiles * args.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      uint32_t s = 0, ph = 0, armed = 0, armed_ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        int g, mt, nt;
        decode_tile(tile, args, g, mt, nt);
        const int m0 = mt * kBM + args.a_row_off;
        const int n0 = nt * kOutN + args.b_row_off;
        const int ga = g * args.a_bmul, gb = g * args.b_bmul;
        for (int kb = 0; kb < args.k_blocks; ++kb) {
          if (!mbar_wait(bar(kBarEmpty + s), ph ^ 1u, abort_flag, err, args.err_site + 1)) {
            ok = false;
            break;
          }
          const uint32_t sa = stage0 + s * kStageBytes, sb = sa + kABytes, fb = bar(kBarFull + s);
          mbar_arrive_expect_tx(fb, kStageBytes);
          armed |= 1u << s;
          armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
          const int k0 = kb * kBK;
          if constexpr (!A_MN) {
            tma_load_3d(sa, &tmA, fb, k0, m0, ga);
          } else {
            tma_load_3d(sa, &tmA, fb, m0, k0, ga);
            tma_load_3d(sa + 8192, &tmA, fb, m0 + 64, k0, ga);
          }
          if constexpr (kGatedB) {
            tma_load_4d(sb, &tmB, fb, k0, n0, 0, g);
            tma_load_4d(sb + 16384, &tmB, fb, k0, n0, 1, g);
          } else if constexpr (!B_MN) {
            tma_load_3d(sb, &tmB, fb, k0, n0, gb);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_3d(sb + 8192 * j, &tmB, fb, n0 + 64 * j, k0, gb);
          }
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        // wait for this CTA's copies still in flight before the CTA exits
        for (int i = 0; i < kStages; ++i)
          if ((armed >> i) & 1u) mbar_wait_drain(bar(kBarFull + i), (armed_ph >> i) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      uint32_t s = 0, ph = 0;
      bool ok = true;
      int it = 0;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
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
          const uint32_t sa = stage0 + s * kStageBytes, sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = A_MN ? sdesc_sw128(sa + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(sb + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(sb + kk * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, kIdesc, static_cast<uint32_t>((kb | kk) != 0));
          }
          umma_commit(bar(kBarEmpty + s));
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(bar(kBarTmemFull + acc));
      }
      // all MMAs this thread issued have completed once the drain barrier flips
      umma_commit(bar(kBarDrain));
      mbar_wait_drain(bar(kBarDrain), 0);
    }
  } else {
    // ---------------- epilogue warps 2..5; TMEM lane quarter = warp % 4
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1) & 1u;
      const bool ok = mbar_wait(bar(kBarTmemFull + acc), use, abort_flag, err, args.err_site + 4);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      int g, mt, nt;
      decode_tile(tile, args, g, mt, nt);
      const uint32_t tacc =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * kBN);
      epilogue_tile<EPI>(args, tacc, g, mt * kBM + row_in_tile, nt * kOutN);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarTmemEmpty + acc));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int EPI, bool A_MN, bool B_MN>
cudaError_t launch_gemm_t(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& args,
                          int grid, cudaStream_t st) {
  auto fn = gemm_kernel<EPI, A_MN, B_MN>;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  fn<<<grid, kThreads, kSmemBytes, st>>>(ta, tb, args);
  return cudaGetLastError();
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
